// Streaming GEMV kernels (M <= 2) for one weight format (see gemv_stream.cuh).
#include "gemv_stream.cuh"

namespace qg {

int stream_launch_q4_k(const DevCtx& dc, const stream::Params& kp, int MT, int LPR, int grid,
                     int warps, int smem, bool pdl, cudaStream_t s) {
    return stream::dispatch<FMT_Q4_K>(dc, kp, MT, LPR, grid, warps, smem, pdl, s);
}

}  // namespace qg
