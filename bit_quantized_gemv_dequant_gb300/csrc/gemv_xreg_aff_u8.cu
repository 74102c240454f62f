// Register-resident-x GEMV instantiations for one weight format (compiled as
// a unit of its own so that the formats build in parallel).
#include "gemv_xreg.cuh"

namespace qg {

int xreg_launch_aff_u8(const DevCtx& dc, const xreg::Params& kp, int MT, int NWC, int grid,
                   int smem, bool pdl, cudaStream_t s) {
    return xreg::dispatch<FMT_AFF_U8>(dc, kp, MT, NWC, grid, smem, pdl, s);
}

}  // namespace qg
