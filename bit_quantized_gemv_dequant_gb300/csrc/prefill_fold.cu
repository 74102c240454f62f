// Affine prefill on the tensor cores with scale and bias folded into the
// weights (QG_OPT_PREFILL_FOLD = 1); the prep kernel and the host side are in
// prefill.cu, the shared pieces in prefill_common.cuh.
#include <algorithm>

#include "prefill_common.cuh"

namespace qg {
namespace prefill {

// Page: qmm_affine.rs (mlx-native 0.21.1), dispatch_qmm_affine_t_f32 and the
// packed 4-bit variant, as for prefill.cu's exact-code kernel. This is the
// opt-in alternative (QG_OPT_PREFILL_FOLD = 1): scale and bias are folded into
// the weights before the tensor cores see them, so a single accumulator in
// tensor memory spans all of K and the epilogue runs once per tile:
//
//     w'[n,k] = fp16_rn( (s[n,g] * q[n,k] + b[n,g]) * 2^f_n ),
//     y[m,n]  = ( sum_k w'[n,k] * xh[m,k] ) * 2^-f_n * 2^-e_m.
//
// f_n puts the row's bound max_g (|s| * qmax + |b|) in [2^14, 2^15), so no
// w' overflows fp16 and every weight above 2^-29 of that bound keeps a
// relative rounding error of at most 2^-11, as xh does. The product error is
// then at most about 2^-10 * sum_k |x w| plus the f32 accumulation: within
// the 2e-3 * sum_k |x w| prefill tolerance. The value s * q + b is formed in
// f32 from the exact code q (2^23 + q through a byte permute, minus 2^23),
// so cancellation between s * q and b costs nothing before the one rounding
// to fp16.
//
//   warps 0-15  converters, then epilogue. Warp w handles weight rows
//               32 * (w % 4) .. + 31 (its tensor-memory lane quarter), the
//               k half (w / 4) % 2 of the 64-wide stages of parity w / 8:
//               codes -> w' in registers -> tcgen05.st into the A buffer.
//               Two warps per lane quarter and stage, and two stages in
//               conversion at once, hide the latency of each stage's chain
//               (barrier wait, shared-memory loads, conversion, tensor-memory
//               store and its wait).
//   warp 16     TMA producer (codes and xh tiles, as in mma_kernel).
//   warps 17-18 MMA issuers: warp 17 + p issues the four K = 16 MMAs of the
//               stages of parity p into accumulator p. A single issuing
//               thread spends a fixed ~0.25 us per stage (barrier wait,
//               commit, first MMA) whatever the MMA size, which made it the
//               bound of the whole tile; two threads on two schedulers halve
//               that. The epilogue adds the two accumulators.
constexpr int kFStages = 8;
constexpr int kFABufs = 8;              // A buffers, 32 columns each
constexpr int kFAcc = 0;                // accumulator p: columns [p * kTileT, (p + 1) * kTileT)
constexpr int kFACol0 = 2 * kTileT;     // A buffers: columns [256, 512)
constexpr int kFConv = 16;              // converter / epilogue warps
constexpr int kFStageWarps = 8;         // converter warps per stage
constexpr int kFProducer = kFConv;
constexpr int kFMma = kFConv + 1;       // and kFMma + 1
constexpr int kFThreads = (kFConv + 3) * 32;
static_assert(kFACol0 + kFABufs * 32 <= kTmemCols, "tensor memory columns");
static_assert(kFStages % 2 == 0, "stage parities own disjoint buffers");
static_assert(kFABufs == kFStages, "stage i uses shared-memory stage and A buffer i % kFStages");

template <bool PACKED>
struct GeoF {
    static constexpr int kStageBytes = StageGeo<PACKED>::kStageBytes;
    static constexpr int kBarOff = kFStages * kStageBytes;
    static constexpr int kSmemBytes = 1024 + kBarOff + 1024;
};

// Four codes (bytes of v) -> 2^23 + q as f32 bit patterns, two pairs.
__device__ __forceinline__ void bytes_to_magic(uint32_t v, float2& q01, float2& q23) {
    q01 = make_float2(__uint_as_float(__byte_perm(v, 0x4B000000u, 0x7440u)),
                      __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7441u)));
    q23 = make_float2(__uint_as_float(__byte_perm(v, 0x4B000000u, 0x7442u)),
                      __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7443u)));
}

// (2^23 + q) pair -> fp16x2 of s * q + b (low half: the first element).
__device__ __forceinline__ uint32_t fold_pair(float2 magic, float2 s2, float2 b2) {
    const float2 q = __fadd2_rn(magic, make_float2(-8388608.f, -8388608.f));  // exact
    const float2 w = __ffma2_rn(s2, q, b2);
    const __half2 hw = __floats2half2_rn(w.x, w.y);
    return *reinterpret_cast<const uint32_t*>(&hw);
}

template <bool PACKED, bool GS16>
__global__ void __launch_bounds__(kFThreads, 1)
    fold_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_x,
                const FoldParams p) {
    using Gm = GeoF<PACKED>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const uint32_t bars = base + Gm::kBarOff;
    auto full = [&](int i) { return bars + 8u * i; };
    auto empty = [&](int i) { return bars + 8u * (kFStages + i); };
    // empty(i): the MMAs of the stage in slot i are done, so both its shared-
    // memory stage and its A buffer may be refilled (one commit frees both).
    auto a_full = [&](int i) { return bars + 8u * (2 * kFStages + i); };
    constexpr int kDone = 3 * kFStages;
    const uint32_t done_bar = bars + 8u * kDone;
    static_assert(8 * (kDone + 1) + 4 <= 1024, "barrier area");
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Gm::kBarOff + 8 * (kDone + 1));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kTileT;
    const int n0 = blockIdx.y * kTileN;
    const int nstages = (p.K + kChunk - 1) / kChunk;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kFStages; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), 1);
        }
        for (int i = 0; i < kFABufs; ++i)
            mbar_init(a_full(i), kFStageWarps);  // one arrival per converter warp
        mbar_init(done_bar, 2);  // one commit per MMA issuer
        fence_mbar_init();
    }
    if (warp == kFMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Everything below reads what the prep kernel wrote (launched as its
    // programmatic dependent, this grid may have started before it finished).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // The next kernel on the stream may become resident now; a dependent
    // launch of it waits for this grid before touching its data.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == kFProducer) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&map_q);
            prefetch_tmap(&map_x);
            int issued = 0;
            for (int i = 0; i < nstages; ++i) {
                const int st = i % kFStages;
                if (i >= kFStages && !mbar_wait_sleep(empty(st), ((i / kFStages) & 1) ^ 1)) {
                    report_error(p.err, DEVERR_TC_WAIT);
                    break;
                }
                const uint32_t sb = base + st * Gm::kStageBytes;
                mbar_arrive_expect_tx(full(st), Gm::kStageBytes);
                tma_load_2d(sb, &map_x, i * kChunk, m0, full(st));
                tma_load_2d(sb + kXhBytes, &map_q, i * StageGeo<PACKED>::kCodeRowBytes, n0, full(st));
                issued = i + 1;
            }
            // Copies must land before the CTA can exit, whatever happened above.
            for (int i = max(0, issued - kFStages); i < issued; ++i)
                if (!mbar_wait(full(i % kFStages), (i / kFStages) & 1))
                    report_error(p.err, DEVERR_WAIT_DRAIN);
        }
    } else if (warp == kFMma || warp == kFMma + 1) {
        // --------------------------------------------------------- MMA issuers
        if (lane == 0) {
            // The loop carries the stage's descriptor and A column as
            // increments (a descriptor's address field is the byte address
            // / 16, and no stage address reaches 2^18).
            const int par = warp - kFMma;
            const uint64_t d0 = sw128_desc(base);
            const uint32_t acc = tmem + kFAcc + par * kTileT, a0 = tmem + kFACol0;
            for (int i = par; i < nstages; i += 2) {
                const int st = i % kFStages;
                // a_full implies the stage's copies landed: the converters waited for them.
                if (!mbar_wait(a_full(st), (uint32_t)(i / kFStages) & 1u)) {
                    report_error(p.err, DEVERR_TC_WAIT);
                    break;
                }
                tc_fence_after();
                const uint64_t d = d0 + (uint64_t)(st * (Gm::kStageBytes >> 4));
                const uint32_t aa = a0 + st * 32;
                tc_mma_ts(acc, aa, d, kIdesc, i > par ? 1u : 0u);
                tc_mma_ts(acc, aa + 8, d + 2, kIdesc, 1u);
                tc_mma_ts(acc, aa + 16, d + 4, kIdesc, 1u);
                tc_mma_ts(acc, aa + 24, d + 6, kIdesc, 1u);
                tc_commit(empty(st));
            }
            tc_commit(done_bar);
            if (!mbar_wait(done_bar, 0)) report_error(p.err, DEVERR_WAIT_DRAIN);
        }
    } else {
        // ------------------------------------------------ converters, epilogue
        const int qd = warp & 3;                   // tensor-memory lane quarter
        const int h = (warp >> 2) & 1;             // k half of each stage
        const int par = warp >> 3;                 // stages of this parity
        const int row = qd * 32 + lane;
        const int n = n0 + row;
        const bool nvalid = n < p.N;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        int f = 0;
        {
            float bm = 0.f;
            if (nvalid)
                for (int j = 0; j < p.GT; ++j) bm = fmaxf(bm, __ldg(p.bpart + (size_t)n * p.GT + j));
            if (bm > 0.f && bm <= 3.402823466e38f) {
                int ex;
                frexpf(bm, &ex);  // bm < 2^ex
                f = min(120, max(-120, 15 - ex));
            }
        }
        const float pw = __int_as_float((127 + f) << 23);
        const float ipw = __int_as_float((127 - f) << 23);
        // Raw scale and bias of the groups of stage i's k half: the first and
        // the second 16 k (the same group unless gs = 16). Column n of the
        // transposed [G, N] arrays: a warp's loads are coalesced.
        auto load_sb = [&](int i, float (&sb4)[4]) {
            const int k0 = i * kChunk + h * 32;
            const int ga = k0 >> p.log2gs;
            const int gb = GS16 ? ga + 1 : ga;
            const bool va = nvalid && ga < p.G, vb = nvalid && gb < p.G;
            sb4[0] = va ? __ldg(p.scales_t + (size_t)ga * p.N + n) : 0.f;
            sb4[1] = va ? __ldg(p.biases_t + (size_t)ga * p.N + n) : 0.f;
            sb4[2] = GS16 ? (vb ? __ldg(p.scales_t + (size_t)gb * p.N + n) : 0.f) : sb4[0];
            sb4[3] = GS16 ? (vb ? __ldg(p.biases_t + (size_t)gb * p.N + n) : 0.f) : sb4[1];
        };
        float nx[4];
        load_sb(par, nx);
        bool ok = true;
        for (int i = par; i < nstages; i += 2) {
            const int st = i % kFStages, ab = st;
            const uint32_t fph = (uint32_t)(i / kFStages) & 1u;
            // Scaled by 2^f only here, one stage after the loads were issued.
            const float2 sA = make_float2(nx[0] * pw, nx[0] * pw), bA = make_float2(nx[1] * pw, nx[1] * pw);
            const float2 sB = make_float2(nx[2] * pw, nx[2] * pw), bB = make_float2(nx[3] * pw, nx[3] * pw);
            if (i + 2 < nstages) load_sb(i + 2, nx);
            if (!warp_wait_sleep(full(st), fph) ||
                (i >= kFStages && !warp_wait_sleep(empty(st), fph ^ 1))) {
                if (lane == 0) report_error(p.err, DEVERR_TC_WAIT);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint8_t* cb = smem + st * Gm::kStageBytes + kXhBytes;
            uint32_t o[16];
            if (!PACKED) {
                // 64-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ ((r >> 1) & 3).
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int c = 2 * h + cc;
                    const uint4 v = *reinterpret_cast<const uint4*>(
                        cb + row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                    const float2 s2 = cc ? sB : sA, b2 = cc ? bB : bA;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float2 q01, q23;
                        bytes_to_magic(w4[e], q01, q23);
                        o[8 * cc + 2 * e] = fold_pair(q01, s2, b2);
                        o[8 * cc + 2 * e + 1] = fold_pair(q23, s2, b2);
                    }
                }
            } else {
                // 32-byte swizzle: chunk c of row r sits at chunk c ^ ((r >> 2) & 1).
                const uint4 v = *reinterpret_cast<const uint4*>(
                    cb + row * 32 + ((h ^ ((row >> 2) & 1)) << 4));
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    // byte i: low nibble = k 8e + 2i, high nibble = k 8e + 2i + 1
                    const uint32_t lo = w4[e] & 0x0F0F0F0Fu;
                    const uint32_t hi = (w4[e] >> 4) & 0x0F0F0F0Fu;
                    const float2 s2 = e < 2 ? sA : sB, b2 = e < 2 ? bA : bB;
                    float2 l01, l23, h01, h23;
                    bytes_to_magic(lo, l01, l23);
                    bytes_to_magic(hi, h01, h23);
                    o[4 * e + 0] = fold_pair(make_float2(l01.x, h01.x), s2, b2);
                    o[4 * e + 1] = fold_pair(make_float2(l01.y, h01.y), s2, b2);
                    o[4 * e + 2] = fold_pair(make_float2(l23.x, h23.x), s2, b2);
                    o[4 * e + 3] = fold_pair(make_float2(l23.y, h23.y), s2, b2);
                }
            }
            tmem_st16(tmem + lane_base + kFACol0 + ab * 32 + h * 16, o);
            tmem_st_wait();
            // One arrival per warp (8 per stage rather than 256 serialised
            // ones), after the fence and the warp barrier that order the
            // warp's tensor-memory stores before it.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full(ab));
        }
        // Epilogue: this warp's 32 activation rows (columns (w / 4) * 32 ..) of its lanes.
        if (ok && warp_wait(done_bar, 0)) {
            tc_fence_after();
            const int c0 = (warp >> 2) * 32;
            // Lane l holds 2^-e of activation row m0 + c0 + l.
            const float ivl = __ldg(p.inv + m0 + c0 + lane);
            float* yp = p.y + (size_t)(m0 + c0) * p.N + (nvalid ? n : 0);
#pragma unroll
            for (int cb16 = 0; cb16 < 2; ++cb16) {
                uint32_t r[16], r1[16];
                tmem_ld16(tmem + lane_base + kFAcc + c0 + cb16 * 16, r);
                // The odd stages' accumulator (never written when K fits one stage).
                if (nstages > 1) {
                    tmem_ld16(tmem + lane_base + kFAcc + kTileT + c0 + cb16 * 16, r1);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) r1[j] = 0u;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int col = cb16 * 16 + j;
                    const float ivm = __shfl_sync(0xFFFFFFFFu, ivl, col);
                    const float a = __uint_as_float(r[j]) + __uint_as_float(r1[j]);
                    if (nvalid && m0 + c0 + col < p.M) yp[(size_t)col * p.N] = (a * ipw) * ivm;
                }
            }
        } else if (ok) {
            if (lane == 0) report_error(p.err, DEVERR_TC_WAIT);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kFMma) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

template <bool PACKED, bool GS16>
int launch_fold(const DevCtx& dc, const CUtensorMap& mq, const CUtensorMap& mx,
                const FoldParams& kp, dim3 grid, cudaStream_t s) {
    constexpr int smem = GeoF<PACKED>::kSmemBytes;
    static int configured[64] = {0};
    auto kern = fold_kernel<PACKED, GS16>;
    if (dc.device >= 0 && dc.device < 64 && !configured[dc.device]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return cuda_fail(e);
        configured[dc.device] = 1;
    }
    // Programmatic dependent of the prep kernel: the prologue (barriers,
    // tensor memory) overlaps the prep's tail.
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mq, mx, kp);
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

int launch_fold_kernel(const DevCtx& dc, bool packed, bool gs16, const CUtensorMap& mq,
                       const CUtensorMap& mx, const FoldParams& fp, dim3 grid, cudaStream_t s) {
    if (gs16)
        return packed ? launch_fold<true, true>(dc, mq, mx, fp, grid, s)
                      : launch_fold<false, true>(dc, mq, mx, fp, grid, s);
    return packed ? launch_fold<true, false>(dc, mq, mx, fp, grid, s)
                  : launch_fold<false, false>(dc, mq, mx, fp, grid, s);
}

int fold_smem_bytes(bool packed) {
    return packed ? GeoF<true>::kSmemBytes : GeoF<false>::kSmemBytes;
}

}  // namespace prefill
}  // namespace qg
