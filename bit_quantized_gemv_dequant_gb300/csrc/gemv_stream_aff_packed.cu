// Streaming GEMV kernels (M <= 2) for one weight format (see gemv_stream.cuh).
#include "gemv_stream.cuh"

namespace qg {

int stream_launch_aff_packed(const DevCtx& dc, const stream::Params& kp, int MT, int LPR, int grid,
                     int warps, int smem, bool pdl, cudaStream_t s) {
    return stream::dispatch<FMT_AFF_PACKED>(dc, kp, MT, LPR, grid, warps, smem, pdl, s);
}

}  // namespace qg
