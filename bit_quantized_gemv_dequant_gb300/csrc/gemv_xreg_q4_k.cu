// Register-resident-x GEMV instantiations for one weight format (compiled as
// a unit of its own so that the formats build in parallel).
#include "gemv_xreg.cuh"

namespace qg {

int xreg_launch_q4_k(const DevCtx& dc, const xreg::Params& kp, int MT, int NWC, int grid,
                   int smem, bool pdl, cudaStream_t s) {
    return xreg::dispatch<FMT_Q4_K>(dc, kp, MT, NWC, grid, smem, pdl, s);
}

}  // namespace qg
