// The register-resident-x kernel (gemv_xreg.cuh) on the prepared AF4-g64
// layout: qmm_af4_g64 with one or two rows of x, planning, the tensor maps
// and the launch. (Slices of four rows were measured slower than the cluster
// kernel of af4_gemv.cu at M = 8: 23.2 against 14.7 us at N = K = 4096.)
//
// Page: qmm_affine.rs (mlx-native 0.21.1), prepare_af4_g64 (the layout) and
// dispatch_qmm_affine_t_packed_simd4_b4_gs64_bf16 (the call). Each 64-row
// block of the plane holds, per 32-group, its 64 rows' 16-byte units side by
// side, so the RC rows of a chunk are one 2-D box: RC x 16 bytes across all
// 32-groups of the block (and RC x 4 bytes across its 64-groups for the
// bf16 scale | bias words).
#include <algorithm>

#include "gemv_xreg.cuh"

namespace qg {
namespace {

template <int MT, int NWC>
int launch_af4(const DevCtx& dc, const xreg::Params& kp, const CUtensorMap& mq,
               const CUtensorMap& mm, int grid, int smem, bool pdl, cudaStream_t s) {
    auto kern = xreg::gemv_xreg_af4_kernel<MT, NWC, xreg::kRPG>;
    static int configured[64] = {0};
    if (dc.device >= 0 && dc.device < 64 && configured[dc.device] < smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             dc.max_smem_optin);
        if (e != cudaSuccess) return cuda_fail(e);
        configured[dc.device] = dc.max_smem_optin;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((NWC + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, kp, mq, mm);
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

bool aligned16p(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Tensor maps of the plane (u8 view [blocks * G32][1024 bytes]) and of the
// metadata ([blocks * G64][256 bytes]) with boxes of RC rows: the plane's
// box carries the 64- (RC = 4) or 128-byte (RC = 8) swizzle that makes the
// consumers' 16-byte reads conflict-free.
int make_maps(const uint32_t* plane, const uint32_t* meta, long long N, long long K, int RC,
              CUtensorMap* mq, CUtensorMap* mm) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    int rc = prefill::encoder(&encode);
    if (rc) return rc;
    const long long units = K / 32, blocks = N / 64;
    {
        const cuuint64_t dims[2] = {1024, (cuuint64_t)(blocks * units)};
        const cuuint64_t strides[1] = {1024};
        const cuuint32_t box[2] = {(cuuint32_t)(RC * 16), (cuuint32_t)units};
        const cuuint32_t es[2] = {1, 1};
        if (encode(mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t*>(plane), dims,
                   strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   RC == 8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return QG_ERR_UNSUPPORTED;
    }
    {
        const cuuint64_t dims[2] = {256, (cuuint64_t)(blocks * (units / 2))};
        const cuuint64_t strides[1] = {256};
        const cuuint32_t box[2] = {(cuuint32_t)(RC * 4), (cuuint32_t)(units / 2)};
        const cuuint32_t es[2] = {1, 1};
        if (encode(mm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t*>(meta), dims,
                   strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return QG_ERR_UNSUPPORTED;
    }
    return QG_OK;
}

}  // namespace

// qmm_af4_g64 on the register-resident-x kernel. Taken for M = 1 and 2 when
// 32-groups fill row groups of 1, 2 or 4 warps (K <= 1024, 2048 or 4096) and
// x, plane and metadata are 16-byte aligned (for both M or for neither, so
// row m of y is the same for M = 1 and 2). Returns QG_ERR_UNSUPPORTED, with
// nothing enqueued, otherwise.
int af4_xreg_launch(const DevCtx& dc, const float* x, const uint32_t* plane,
                    const uint32_t* meta, float* y, long long M, long long N, long long K,
                    cudaStream_t s) {
    if (launch_option(QG_OPT_XREG) == 0 || M < 1 || M > 2) return QG_ERR_UNSUPPORTED;
    if (K % 64 || N % 64 || N > (1ll << 30)) return QG_ERR_UNSUPPORTED;
    const long long units = K / 32;
    const long long WG = (units + 31) / 32;
    if (WG != 1 && WG != 2 && WG != 4) return QG_ERR_UNSUPPORTED;
    if (!aligned16p(x) || !aligned16p(plane) || !aligned16p(meta)) return QG_ERR_UNSUPPORTED;

    const long long pdl_mode = launch_option(QG_OPT_PDL);
    const long long want_w = launch_option(QG_OPT_XREG_WARPS);
    // CTAs per call: for independent calls (QG_OPT_PDL = 2) on the automatic
    // four-warp shape, whose CTAs share SMs with the neighbouring calls', one
    // per two SMs (M = 1, N = K = 4096, long runs: 2.00 us against 2.02 with
    // three per four and 2.06 with one per SM); else one per SM, unless
    // QG_OPT_XREG_CTAS sets it.
    const long long ctas_opt = launch_option(QG_OPT_XREG_CTAS);
    const long long quads = N / 4;
    const long long grid_max = ctas_opt > 0 ? (long long)dc.num_sms * ctas_opt
                               : (pdl_mode == 2 && want_w == 0)
                                   ? std::max<long long>(1, dc.num_sms / 2)
                                   : (long long)dc.num_sms;
    const long long grid = std::min<long long>(quads, grid_max);
    const long long rows_cta = 4 * ((quads + grid - 1) / grid);

    // Plan every slice before anything is enqueued.
    struct Slice {
        int Mc, MT, NWC, NRG, RC, S, smem, rbuf, red_floats, slot, code_bytes;
    };
    Slice sl[4];
    int ns = 0;
    const int step = M <= 2 ? 2 : 4;
    for (long long m0 = 0; m0 < M; m0 += step, ++ns) {
        Slice& q = sl[ns];
        q.Mc = (int)std::min<long long>(step, M - m0);
        q.MT = q.Mc <= 2 ? q.Mc : 4;
        q.NWC = 8;
        if (q.MT == 4) {
            q.NWC = 4;
        } else if (want_w != 0) {
            if (want_w % WG == 0 && !(want_w == 16 && q.MT == 2)) q.NWC = (int)want_w;
        } else if (pdl_mode == 2) {
            q.NWC = 4;
        }
        // At most two row groups: chunks of 4 or 8 rows (the swizzled box).
        q.NRG = (int)std::min<long long>(2, q.NWC / WG);
        q.RC = q.NRG * xreg::kRPG;
        const long long code_bytes = (long long)q.RC * 16 * units;
        const long long slot =
            ((code_bytes + (long long)q.RC * 4 * (units / 2)) + 1023) & ~1023ll;
        const long long rbuf =
            std::max<long long>(q.RC, std::min<long long>(rows_cta, 4096 / (q.MT * WG)));
        const long long red_floats = (rbuf * q.MT * WG + 3) & ~3ll;
        const long long fixed =
            (red_floats + (long long)q.MT * K) * 4 + (long long)q.NWC * q.MT * 4 + 128;
        const bool co = ((q.NWC == 8 || q.NWC == 12) && q.MT == 1) || (q.NWC == 4 && q.MT <= 2);
        const int per_sm = q.NWC == 4 ? (q.MT == 1 ? 4 : 3) : 2;
        long long budget =
            (co ? (long long)dc.smem_per_sm / per_sm - dc.reserved_smem : dc.max_smem_optin) - 1024;
        long long S = std::min<long long>(16, (budget - fixed) / (slot + 16));
        if (S < 2) {
            budget = dc.max_smem_optin - 1024;
            S = std::min<long long>(16, (budget - fixed) / (slot + 16));
        }
        if (S < 2) return QG_ERR_UNSUPPORTED;
        q.S = (int)S;
        q.smem = (int)(S * (slot + 16) + fixed - 128 + 1024);
        q.rbuf = (int)rbuf;
        q.red_floats = (int)red_floats;
        q.slot = (int)slot;
        q.code_bytes = (int)code_bytes;
    }

    CUtensorMap maps[2][2];  // [RC == 8][plane, metadata]
    bool made[2] = {false, false};
    for (int i = 0; i < ns; ++i) {
        const int which = sl[i].RC == 8 ? 1 : 0;
        if (!made[which]) {
            const int rc = make_maps(plane, meta, N, K, sl[i].RC, &maps[which][0], &maps[which][1]);
            if (rc) return rc;
            made[which] = true;
        }
    }
    const bool pdl = pdl_mode != 0;
    for (int i = 0; i < ns; ++i) {
        const Slice& q = sl[i];
        const long long m0 = (long long)i * step;
        xreg::Params kp{};
        kp.w[0] = kp.w[1] = reinterpret_cast<const uint8_t*>(plane);
        kp.out[0] = kp.out[1] = y + m0 * N;
        kp.x = x + m0 * K;
        kp.M = q.Mc;
        kp.N = (int)N;
        kp.K = (int)K;
        kp.nw = 1;
        kp.rows_base = (int)(quads / grid);
        kp.rows_rem = (int)(quads % grid);
        kp.row_unit = 4;
        kp.S = q.S;
        kp.slot_bytes = q.slot;
        kp.sb_off = q.code_bytes;
        kp.WG = (int)WG;
        kp.NRG = q.NRG;
        kp.RC = q.RC;
        kp.units = (int)units;
        kp.rbuf = q.rbuf;
        kp.red_floats = q.red_floats;
        kp.ahead = 0;
        kp.dep_wait = pdl_mode == 2 ? 0 : 1;
        kp.err = dc.err;
        const int which = q.RC == 8 ? 1 : 0;
        const CUtensorMap& mq = maps[which][0];
        const CUtensorMap& mm = maps[which][1];
        const int g = (int)grid;
        int rc;
        if (q.MT == 1)
            rc = q.NWC == 4   ? launch_af4<1, 4>(dc, kp, mq, mm, g, q.smem, pdl, s)
                 : q.NWC == 8 ? launch_af4<1, 8>(dc, kp, mq, mm, g, q.smem, pdl, s)
                              : launch_af4<1, 16>(dc, kp, mq, mm, g, q.smem, pdl, s);
        else
            rc = q.NWC == 4 ? launch_af4<2, 4>(dc, kp, mq, mm, g, q.smem, pdl, s)
                            : launch_af4<2, 8>(dc, kp, mq, mm, g, q.smem, pdl, s);
        if (rc != QG_OK) return rc;
    }
    return QG_OK;
}

}  // namespace qg
