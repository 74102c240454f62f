// Fast GEMV kernels for one weight format (see gemv_fast.cuh).
#include "gemv_fast.cuh"

namespace qg {

int fast_launch_aff_packed(const DevCtx& dc, const fast::Params& kp, int MT, int R, int GW, int W, int grid,
                   int smem, bool pdl, cudaStream_t s) {
    return fast::dispatch<FMT_AFF_PACKED>(dc, kp, MT, R, GW, W, grid, smem, pdl, s);
}

}  // namespace qg
