// Affine-quantized matmul for many activation rows (prefill) on the fifth-
// generation tensor cores: the prep kernel, the exact-code kernel (the
// default) and the host side of both kernels. The folded-weight kernel
// (QG_OPT_PREFILL_FOLD = 1) is in prefill_fold.cu, the pieces both share in
// prefill_common.cuh.
//
// Page: qmm_affine.rs (mlx-native 0.21.1), dispatch_qmm_affine_t_f32 and the
// packed 4-bit variant: y[m,n] = sum_k x[m,k] * w[n,k], w[n,k] = s[n,g] *
// q[n,k] + b[n,g], g = k / gs. Regrouping the sum per quantization group,
//
//     y[m,n] = sum_g ( s[n,g] * P_g[n,m] + b[n,g] * X_g[m] ),
//     P_g[n,m] = sum_{k in g} q[n,k] * x[m,k],   X_g[m] = sum_{k in g} x[m,k],
//
// the inner sums P_g are a plain integer-weight contraction, which runs here
// as tcgen05 MMAs: the codes q (integers 0..255) are exact in fp16, and x is
// rounded to fp16 once. The same page's bf16 table-plus-sums kernels (the
// K9/K10 section) split the sum the same way; this kernel keeps the integer
// codes exact and applies scale and bias in an f32 epilogue.
//
// Two launches per call:
//   prep: for each activation row m, a power-of-two scale 2^e_m (so that the
//         largest |x| lands in [2^14, 2^15) and fp16 neither overflows nor
//         goes subnormal early), xh = fp16_rn(x * 2^e_m), and X_g[m] summed in
//         f32 from the ROUNDED values. Using the rounded values in both terms
//         makes the factored sum equal sum_k w * xh up to f32 rounding, so the
//         error is at most 2^-11 * sum_k |w * x| plus f32 rounding.
//   main: one CTA per (128 weight rows) x (128 activation rows) tile.
//         warp 12      TMA producer: per 64-wide k sub-stage, the code tile
//                      (128 rows, u8 or packed) and the xh tile (128 rows,
//                      fp16, 128-byte swizzle) into a ring of sub-stages;
//                      two sub-stages (a 128-wide step) complete on one
//                      barrier.
//         warps 0-3    converters: codes -> fp16 (exact) in registers, stored
//                      into tensor memory as the A operand (tcgen05.st); the
//                      converted weights never pass through shared memory.
//                      One A buffer (64 columns) per step, two buffers.
//         warp 13      MMA issuer: kind::f16, M=128 (weight rows), N=128
//                      (activation rows), K=16 per instruction, eight per
//                      step, f32 accumulators P_g in tensor memory, three
//                      buffers; it waits for the epilogue to release a P
//                      buffer before a group starts in it.
//         warps 4-11   epilogue: acc += s * P_g + b * X_g per group, in f32
//                      registers (scales and biases read four groups
//                      ahead); at the end y = acc * 2^-e_m.
//       Every barrier wait, fence and commit of the converters and the MMA
//       thread is paid once per 128-wide step: measured, these hand-offs, not
//       the copies or the arithmetic, bounded the kernel with 64-wide ones.
// Every wait is bounded; a wait that runs out records an error bit and the
// CTA winds down (drains its copies and MMAs, frees tensor memory) instead of
// hanging.
#include <algorithm>
#include <mutex>

#include "prefill_common.cuh"

namespace qg {
namespace prefill {

constexpr int kStages = 8;     // 64-wide sub-stages in the shared-memory ring
constexpr int kSteps = kStages / 2;  // 128-wide steps: two sub-stages per barrier
constexpr int kABufs = 2;      // A operand buffers in tensor memory (64 columns each)
constexpr int kPBufs = 3;      // P_g accumulators in tensor memory
constexpr int kPCols = kTileT; // columns per P buffer
constexpr int kACol0 = kPBufs * kPCols;  // A buffers follow: 384 + 2 * 64 = 512 columns
constexpr int kXSlots = 32;    // ring of per-group activation sums in shared memory
constexpr int kXSlotBytes = kTileT * 4;
constexpr int kEpiWarps = 8;  // epilogue warps 4 .. 4 + kEpiWarps - 1
constexpr int kEpiCols = kTileT / (kEpiWarps / 4);  // activation rows (columns) per epilogue warp
constexpr int kProducerWarp = 4 + kEpiWarps;
constexpr int kMmaWarp = 5 + kEpiWarps;
constexpr int kThreads = (6 + kEpiWarps) * 32;

struct Params {
    const float* scales_t; // [G, N] (scales transposed by the prep kernel)
    const float* biases_t; // [G, N]
    float* y;              // [M, N]
    const float* xsum;     // [G, Mp] group sums of the rounded activations
    const float* inv;      // [Mp] 2^-e_m
    int M, N, K, G, Mp;
    int gs;                // group size
    int spgs;              // 128-wide steps per group when gs >= 128 (else 1)
    unsigned* err;
};

template <bool PACKED>
struct Geo : StageGeo<PACKED> {
    static constexpr int kXOff = kStages * StageGeo<PACKED>::kStageBytes;
    static constexpr int kBarOff = kXOff + kXSlots * kXSlotBytes;
    static constexpr int kSmemBytes = 1024 + kBarOff + 1024;
};

// Four u8 codes (little-endian bytes of v) -> two fp16x2 words holding the
// exact values: 0x64 above each byte is 1024 + q, minus 1024 leaves q.
__device__ __forceinline__ void codes4_to_h2(uint32_t v, uint32_t& lo, uint32_t& hi) {
    const uint32_t a = __byte_perm(v, 0x6464u, 0x4140u);
    const uint32_t b = __byte_perm(v, 0x6464u, 0x4342u);
    asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64006400u));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64006400u));
}

// ------------------------------------------------------------- prep kernel
// Blocks [0, Mp) prepare activation rows (with xsum = nullptr, no group
// sums). The blocks after them transpose 32 x 32 tiles of the scales and
// biases to [G, N], so that a kernel handling one weight row per thread reads
// them coalesced; with bpart given they also write, per weight row and tile,
// the bound max_g (|s| * qmax + |b|) over the tile's 32 groups
// (bpart[n * ceil(G / 32) + tile]) for fold_kernel.
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(
    const float* __restrict__ x, __half* __restrict__ xh, float* __restrict__ xsum,
    float* __restrict__ inv, const float* __restrict__ sc, const float* __restrict__ bi,
    float* __restrict__ sc_t, float* __restrict__ bi_t, float* __restrict__ bpart, float qmax,
    int M, int N, int K, int gs, int G, int Mp) {
    __shared__ float red[kPrepThreads / 32];
    __shared__ float amax_s;
    __shared__ float tile[2][32][33];
    const int t = threadIdx.x;
    // This kernel is launched as a programmatic dependent of whatever precedes
    // it on the stream (it may be resident before that kernel ends): it waits
    // for it before reading or writing anything. fold_kernel, launched as this
    // kernel's dependent, may then start its prologue; it waits for this grid
    // before reading what it writes.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if ((int)blockIdx.x >= Mp) {
        const int tiles_g = (G + 31) / 32;
        const int tb = blockIdx.x - Mp;
        const int n_0 = (tb / tiles_g) * 32, g_0 = (tb % tiles_g) * 32;
        const int tx = t & 31, ty = t >> 5;  // 32 x 8 threads
        for (int r = ty; r < 32; r += 8) {
            const int n = n_0 + r, g = g_0 + tx;
            const bool in = n < N && g < G;
            const float sv = in ? __ldg(sc + (size_t)n * G + g) : 0.f;
            const float bv = in ? __ldg(bi + (size_t)n * G + g) : 0.f;
            tile[0][r][tx] = sv;
            tile[1][r][tx] = bv;
            if (bpart) {
                float mx = fmaf(fabsf(sv), qmax, fabsf(bv));
#pragma unroll
                for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
                if (tx == 0 && n < N) bpart[(size_t)n * tiles_g + g_0 / 32] = mx;
            }
        }
        __syncthreads();
        for (int r = ty; r < 32; r += 8) {
            const int g = g_0 + r, n = n_0 + tx;
            if (g < G && n < N) {
                sc_t[(size_t)g * N + n] = tile[0][tx][r];
                bi_t[(size_t)g * N + n] = tile[1][tx][r];
            }
        }
        return;
    }
    const int m = blockIdx.x;
    const int lane = t & 31, warp = t >> 5;
    if (m >= M) {  // padding rows: zero group sums so the epilogue reads defined values
        if (xsum)
            for (int g = t; g < G; g += kPrepThreads) xsum[(size_t)g * Mp + m] = 0.f;
        if (t == 0) inv[m] = 1.f;
        return;
    }
    const float4* xr = reinterpret_cast<const float4*>(x + (size_t)m * K);
    const int quads = K >> 2;
    // Rows of up to kCacheQ * 1024 floats stay in registers between the two
    // passes (one read of x); longer rows are read twice.
    constexpr int kCacheQ = 8;
    const bool cached = quads <= kCacheQ * kPrepThreads;
    float4 cache[kCacheQ];
    float amax = 0.f;
    auto amax4 = [](float4 v) {
        return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    };
    if (cached) {
#pragma unroll
        for (int j = 0; j < kCacheQ; ++j) {
            const int c = t + j * kPrepThreads;
            cache[j] = c < quads ? __ldg(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            amax = fmaxf(amax, amax4(cache[j]));
        }
    } else {
        for (int c = t; c < quads; c += kPrepThreads) amax = fmaxf(amax, amax4(__ldg(xr + c)));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    if (t == 0) {
        float a = red[0];
        for (int w = 1; w < kPrepThreads / 32; ++w) a = fmaxf(a, red[w]);
        amax_s = a;
    }
    __syncthreads();
    amax = amax_s;
    int e = 0;
    if (amax > 0.f && amax <= 3.402823466e38f) {
        int ex;
        frexpf(amax, &ex);         // amax = f * 2^ex, f in [0.5, 1)
        e = min(126, max(-126, 15 - ex));
    }
    const float scale = ldexpf(1.f, e);
    if (t == 0) inv[m] = ldexpf(1.f, -e);
    __syncthreads();  // red[] is reused below

    // Threads t .. t + gs/4 - 1 of one pass hold one group (1024 = 4 * 256 is a
    // multiple of every gs <= 1024, so a group never straddles two passes).
    const int width = min(gs >> 2, 32);
    const int groups_per_pass = (4 * kPrepThreads) / gs;  // 0 when gs > 1024 (not allowed)
    __half2* xo = reinterpret_cast<__half2*>(xh + (size_t)m * K);
    // One pass of kPrepThreads float4s starting at element 4 * base; v is this
    // thread's float4 (ignored past the row's end).
    auto pass = [&](int base, float4 v) {
        const int c = base + t;
        float f = 0.f;
        if (c < quads) {
            const __half2 h0 = __floats2half2_rn(v.x * scale, v.y * scale);
            const __half2 h1 = __floats2half2_rn(v.z * scale, v.w * scale);
            xo[2 * c] = h0;
            xo[2 * c + 1] = h1;
            const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
            f = (f0.x + f0.y) + (f1.x + f1.y);
        }
        for (int o = width >> 1; o; o >>= 1) f += __shfl_xor_sync(0xFFFFFFFFu, f, o);
        if ((gs >> 2) <= 32) {
            if (xsum && (lane & (width - 1)) == 0 && c < quads) {
                const int g = (c << 2) >> (__ffs(gs) - 1);
                xsum[(size_t)g * Mp + m] = f;
            }
        } else {
            if (lane == 0) red[warp] = f;
            __syncthreads();
            const int wpg = gs >> 7;  // warps per group
            if (t < groups_per_pass) {
                float s = 0.f;
                for (int w = 0; w < wpg; ++w) s += red[t * wpg + w];
                const int g = base / (gs >> 2) + t;
                if (xsum && g < G) xsum[(size_t)g * Mp + m] = s;
            }
            __syncthreads();
        }
    };
    if (cached) {
#pragma unroll
        for (int j = 0; j < kCacheQ; ++j) {
            if (j * kPrepThreads >= quads) break;  // uniform over the block
            pass(j * kPrepThreads, cache[j]);
        }
    } else {
        for (int base = 0; base < quads; base += kPrepThreads) {
            const int c = base + t;
            pass(base, c < quads ? __ldg(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f));
        }
    }
}

// ------------------------------------------------------------- main kernel
// GK: MMA k-steps (16 wide) per group when a group fits in one 128-wide step
// (gs = 16, 32, 64 -> 1, 2, 4), or 8 when a group spans whole steps (gs >= 128).
template <bool PACKED, int GK>
__global__ void __launch_bounds__(kThreads, 1)
    mma_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_x,
               const Params p) {
    using Gm = Geo<PACKED>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const uint32_t bars = base + Gm::kBarOff;
    auto full = [&](int i) { return bars + 8u * i; };
    auto empty = [&](int i) { return bars + 8u * (kStages + i); };
    auto a_full = [&](int i) { return bars + 8u * (2 * kStages + i); };
    auto a_empty = [&](int i) { return bars + 8u * (2 * kStages + kABufs + i); };
    constexpr int kPB = 2 * kStages + 2 * kABufs;   // first P barrier
    constexpr int kXB = kPB + 2 * kPBufs;            // first activation-sum barrier
    constexpr int kDone = kXB + 2 * kXSlots;
    auto p_full = [&](int i) { return bars + 8u * (kPB + i); };
    auto p_empty = [&](int i) { return bars + 8u * (kPB + kPBufs + i); };
    auto x_full = [&](int i) { return bars + 8u * (kXB + i); };
    auto x_empty = [&](int i) { return bars + 8u * (kXB + kXSlots + i); };
    const uint32_t done_bar = bars + 8u * kDone;
    static_assert(8 * (kDone + 1) + 4 <= 1024, "barrier area");
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Gm::kBarOff + 8 * (kDone + 1));
    const uint32_t xring = base + Gm::kXOff;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kTileT;
    const int n0 = blockIdx.y * kTileN;
    const int nsub = (p.K + kChunk - 1) / kChunk;            // 64-wide sub-stages
    const int nsteps = (nsub + 1) / 2;                         // 128-wide steps
    const int nks = p.K >> 4;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSteps; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), 1);
        }
        for (int i = 0; i < kABufs; ++i) {
            mbar_init(a_full(i), 4);  // one arrival per converter warp
            mbar_init(a_empty(i), 1);
        }
        for (int i = 0; i < kPBufs; ++i) {
            mbar_init(p_full(i), 1);
            mbar_init(p_empty(i), kEpiWarps);  // one arrival per epilogue warp
        }
        for (int i = 0; i < kXSlots; ++i) {
            mbar_init(x_full(i), 1);
            mbar_init(x_empty(i), kEpiWarps);
        }
        mbar_init(done_bar, 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
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

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&map_q);
            prefetch_tmap(&map_x);
            int issued = 0, xissued = 0;
            bool dead = false;
            for (int i = 0; i < nsteps && !dead; ++i) {
                const int t = i % kSteps;
                if (i >= kSteps && !mbar_wait(empty(t), ((i / kSteps) & 1) ^ 1)) {
                    report_error(p.err, DEVERR_TC_WAIT);
                    break;
                }
                // Step i: sub-stages 2i and 2i + 1 (the last step of a K
                // that is an odd number of 64s has one) in ring regions 2t, 2t + 1.
                const int ns = min(2, nsub - 2 * i);
                mbar_arrive_expect_tx(full(t), (uint32_t)(ns * Gm::kStageBytes));
                for (int sub = 0; sub < ns; ++sub) {
                    const uint32_t sb = base + (2 * t + sub) * Gm::kStageBytes;
                    tma_load_2d(sb, &map_x, (2 * i + sub) * kChunk, m0, full(t));
                    tma_load_2d(sb + kXhBytes, &map_q, (2 * i + sub) * Gm::kCodeRowBytes, n0,
                                full(t));
                }
                issued = i + 1;
                // Activation sums of the groups that start inside this step.
                const int ke = min(p.K, (i + 1) * 2 * kChunk);
                for (int j = xissued; j * p.gs < ke; ++j) {
                    const int sl = j % kXSlots;
                    if (j >= kXSlots && !mbar_wait(x_empty(sl), ((j / kXSlots) & 1) ^ 1)) {
                        report_error(p.err, DEVERR_TC_WAIT);
                        dead = true;
                        break;
                    }
                    mbar_arrive_expect_tx(x_full(sl), kXSlotBytes);
                    bulk_g2s_nohint(xring + sl * kXSlotBytes, p.xsum + (size_t)j * p.Mp + m0,
                                    kXSlotBytes, x_full(sl));
                    xissued = j + 1;
                }
            }
            // Copies must land before the CTA can exit, whatever happened above.
            for (int i = max(0, issued - kSteps); i < issued; ++i)
                if (!mbar_wait(full(i % kSteps), (i / kSteps) & 1))
                    report_error(p.err, DEVERR_WAIT_DRAIN);
            for (int j = max(0, xissued - kXSlots); j < xissued; ++j)
                if (!mbar_wait(x_full(j % kXSlots), (j / kXSlots) & 1))
                    report_error(p.err, DEVERR_WAIT_DRAIN);
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------- MMA issuer
        // The issue loop is kept lean (ring indices and phase bits carried in
        // counters, k-steps unrolled): every instruction between two MMAs
        // of the single issuing thread delays the tensor pipe.
        if (lane == 0) {
            int t = 0, ab = 0, pb = 0, gst = 0, groups = 0;
            uint32_t aph = 0, pph = 0;
            bool dead = false;
            for (int i = 0; i < nsteps && !dead; ++i) {
                const int nk = min(8, nks - 8 * i);
                // a_full implies the step's copies landed (the converters
                // waited for them): one barrier poll per 128-wide step.
                if (!mbar_wait(a_full(ab), aph)) {
                    report_error(p.err, DEVERR_TC_WAIT);
                    break;
                }
                tc_fence_after();
                const uint32_t sb0 = base + (2 * t) * Gm::kStageBytes;
                const uint32_t aa = tmem + kACol0 + ab * 64;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    if (kk >= nk) break;
                    const bool gstart = (GK == 8) ? (kk == 0 && gst == 0) : (kk % GK == 0);
                    // A group's P buffer must have been drained by the epilogue.
                    if (gstart && groups >= kPBufs) {
                        if (!mbar_wait(p_empty(pb), pph ^ 1)) {
                            report_error(p.err, DEVERR_TC_WAIT);
                            dead = true;
                            break;
                        }
                        tc_fence_after();
                    }
                    tc_mma_ts(tmem + pb * kPCols, aa + kk * 8,
                              sw128_desc(sb0 + (kk >> 2) * Gm::kStageBytes + (kk & 3) * 32), kIdesc,
                              gstart ? 0u : 1u);
                    const bool gend =
                        (GK == 8) ? (kk == 7 && gst == p.spgs - 1) : (kk % GK == GK - 1);
                    if (gend) {
                        tc_commit(p_full(pb));
                        ++groups;
                        if (++pb == kPBufs) { pb = 0; pph ^= 1; }
                    }
                }
                tc_commit(empty(t));
                tc_commit(a_empty(ab));
                if (++t == kSteps) t = 0;
                if (++ab == kABufs) { ab = 0; aph ^= 1; }
                if (GK == 8 && ++gst == p.spgs) gst = 0;
            }
            tc_commit(done_bar);
            if (!mbar_wait(done_bar, 0)) report_error(p.err, DEVERR_WAIT_DRAIN);
        }
    } else if (warp < 4) {
        // ---------------------------------------------------------- converters
        const int row = threadIdx.x;  // 0..127: lane 32*warp + lane of tensor memory
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        int t = 0, ab = 0;
        uint32_t fph = 0, aph = 0;
        for (int i = 0; i < nsteps; ++i) {
            if (!warp_wait(full(t), fph) || (i >= kABufs && !warp_wait(a_empty(ab), aph ^ 1))) {
                if (lane == 0) report_error(p.err, DEVERR_TC_WAIT);
                break;
            }
            tc_fence_after();
            const int ns = min(2, nsub - 2 * i);
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
                if (sub >= ns) break;
                const uint8_t* cb = smem + (2 * t + sub) * Gm::kStageBytes + kXhBytes;
                const uint32_t acol = tmem + lane_base + kACol0 + ab * 64 + sub * 32;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t h[16];
                    if (!PACKED) {
                        // 64-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ ((r >> 1) & 3).
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            const int c = 2 * hf + cc;
                            const uint4 v = *reinterpret_cast<const uint4*>(
                                cb + row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
                            codes4_to_h2(v.x, h[8 * cc + 0], h[8 * cc + 1]);
                            codes4_to_h2(v.y, h[8 * cc + 2], h[8 * cc + 3]);
                            codes4_to_h2(v.z, h[8 * cc + 4], h[8 * cc + 5]);
                            codes4_to_h2(v.w, h[8 * cc + 6], h[8 * cc + 7]);
                        }
                    } else {
                        // 32-byte swizzle: chunk c of row r sits at chunk c ^ ((r >> 2) & 1).
                        const uint4 v = *reinterpret_cast<const uint4*>(
                            cb + row * 32 + ((hf ^ ((row >> 2) & 1)) << 4));
                        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            // low nibble of each byte = even k, high nibble = odd k
                            const uint32_t lo = w4[e] & 0x0F0F0F0Fu;
                            const uint32_t hi = (w4[e] >> 4) & 0x0F0F0F0Fu;
                            codes4_to_h2(__byte_perm(lo, hi, 0x5140u), h[4 * e + 0], h[4 * e + 1]);
                            codes4_to_h2(__byte_perm(lo, hi, 0x7362u), h[4 * e + 2], h[4 * e + 3]);
                        }
                    }
                    tmem_st16(acol + hf * 16, h);
                }
            }
            tmem_st_wait();
            // One arrival per warp: the barrier sees 4 arrivals instead of 128
            // serialised ones. The warp's tensor-memory stores are ordered
            // before it by the fence and the warp barrier.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full(ab));
            if (++t == kSteps) { t = 0; fph ^= 1; }
            if (++ab == kABufs) { ab = 0; aph ^= 1; }
        }
    } else if (warp < 4 + kEpiWarps) {
        // ------------------------------------------------------------ epilogue
        constexpr int kChunks = kEpiCols / 16;   // 16-column tensor-memory loads per group
        const int q = warp & 3;                  // tensor-memory lane quarter
        const int part = (warp - 4) >> 2;        // which kEpiCols activation rows
        const int n = n0 + q * 32 + lane;
        const bool nvalid = n < p.N;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const int t0 = m0 + part * kEpiCols;
        float2 acc[kEpiCols / 2];
#pragma unroll
        for (int c = 0; c < kEpiCols / 2; ++c) acc[c] = make_float2(0.f, 0.f);
        bool ok = true;
        // Column n of the transposed scales/biases: a warp's loads are coalesced.
        const float* srow = p.scales_t + (nvalid ? n : 0);
        const float* brow = p.biases_t + (nvalid ? n : 0);
        int pb = 0, xsl = 0;
        uint32_t pph = 0, xph = 0;
        // Scales and biases are loaded kAhead groups ahead (a group takes well
        // under an L2 round trip), in a register queue shifted once per group.
        constexpr int kAhead = 4;
        float sq[kAhead], bq[kAhead];
#pragma unroll
        for (int u = 0; u < kAhead; ++u) {
            sq[u] = (nvalid && u < p.G) ? __ldg(srow + (size_t)u * p.N) : 0.f;
            bq[u] = (nvalid && u < p.G) ? __ldg(brow + (size_t)u * p.N) : 0.f;
        }
        // acc[c] (tokens 2c, 2c+1 of this warp's kEpiCols) += s * P + b * X for
        // one 16-column chunk hf of P.
        auto fma_chunk = [&](int hf, const uint32_t (&r)[16], const float4 (&xv)[4], float2 s2,
                             float2 b2) {
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const int c = hf * 8 + c4 * 2;
                float2 t = __ffma2_rn(b2, make_float2(xv[c4].x, xv[c4].y), acc[c]);
                acc[c] = __ffma2_rn(s2, make_float2(__uint_as_float(r[4 * c4]),
                                                    __uint_as_float(r[4 * c4 + 1])), t);
                t = __ffma2_rn(b2, make_float2(xv[c4].z, xv[c4].w), acc[c + 1]);
                acc[c + 1] = __ffma2_rn(s2, make_float2(__uint_as_float(r[4 * c4 + 2]),
                                                        __uint_as_float(r[4 * c4 + 3])), t);
            }
        };
        for (int j = 0; j < p.G; ++j) {
            const float2 s2 = make_float2(sq[0], sq[0]), b2 = make_float2(bq[0], bq[0]);
#pragma unroll
            for (int u = 0; u + 1 < kAhead; ++u) {
                sq[u] = sq[u + 1];
                bq[u] = bq[u + 1];
            }
            const bool more = nvalid && j + kAhead < p.G;
            sq[kAhead - 1] = more ? __ldg(srow + (size_t)(j + kAhead) * p.N) : 0.f;
            bq[kAhead - 1] = more ? __ldg(brow + (size_t)(j + kAhead) * p.N) : 0.f;
            if (!warp_wait(p_full(pb), pph) || !warp_wait(x_full(xsl), xph)) {
                if (lane == 0) report_error(p.err, DEVERR_TC_WAIT);
                ok = false;
                break;
            }
            tc_fence_after();
            const float4* xs = reinterpret_cast<const float4*>(smem + Gm::kXOff + xsl * kXSlotBytes) +
                               part * (kEpiCols / 4);
            const uint32_t pcol = tmem + lane_base + pb * kPCols + part * kEpiCols;
            // 16-column chunks; the load of chunk hf+1 is in flight while chunk hf
            // is multiplied.
            uint32_t ra[16], rb[16];
            float4 xv[4];
            tmem_ld16_async(pcol, ra);
            tmem_wait16(ra);
#pragma unroll
            for (int hf = 0; hf < kChunks; ++hf) {
                uint32_t(&cur)[16] = (hf & 1) ? rb : ra;
                uint32_t(&nxt)[16] = (hf & 1) ? ra : rb;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) xv[c4] = xs[4 * hf + c4];
                if (hf + 1 < kChunks) tmem_ld16_async(pcol + 16 * (hf + 1), nxt);
                if (hf + 1 == kChunks) {
                    // Everything of group j is read: release P and the sums.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(p_empty(pb));
                        mbar_arrive(x_empty(xsl));
                    }
                }
                fma_chunk(hf, cur, xv, s2, b2);
                if (hf + 1 < kChunks) tmem_wait16(nxt);
            }
            if (++pb == kPBufs) { pb = 0; pph ^= 1; }
            if (++xsl == kXSlots) { xsl = 0; xph ^= 1; }
        }
        if (ok) {
            // Lane l < kEpiCols / 2 holds 2^-e of activation rows t0 + 2l, t0 + 2l + 1.
            const float2 iv = lane < kEpiCols / 2
                                  ? __ldg(reinterpret_cast<const float2*>(p.inv + t0) + lane)
                                  : make_float2(1.f, 1.f);
            float* yp = p.y + (size_t)t0 * p.N + (nvalid ? n : 0);
#pragma unroll
            for (int c = 0; c < kEpiCols / 2; ++c) {
                const float2 sc = make_float2(__shfl_sync(0xFFFFFFFFu, iv.x, c),
                                              __shfl_sync(0xFFFFFFFFu, iv.y, c));
                const int m = t0 + 2 * c;
                if (nvalid && m < p.M) *yp = acc[c].x * sc.x;
                yp += p.N;
                if (nvalid && m + 1 < p.M) *yp = acc[c].y * sc.y;
                yp += p.N;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ------------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_rc = cudaSuccess;

int encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        g_encode_rc = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                       cudaEnableDefault, &q);
        if (g_encode_rc == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (g_encode_rc != cudaSuccess) return cuda_fail(g_encode_rc);
    if (!g_encode) return QG_ERR_UNSUPPORTED;
    *out = g_encode;
    return QG_OK;
}

struct Layout {
    size_t xh, xsum, inv, sc_t, bi_t, bpart, total;
    int Mp, G;
};

Layout layout(const GemvArgs& a) {
    Layout L{};
    L.Mp = (int)((a.M + kTileT - 1) / kTileT * kTileT);
    L.G = (int)(a.K / a.gs);
    auto up = [](size_t v) { return (v + 1023) & ~(size_t)1023; };
    L.xh = 0;
    L.xsum = up((size_t)a.M * a.K * 2);
    L.inv = L.xsum + up((size_t)L.G * L.Mp * 4);
    L.sc_t = L.inv + up((size_t)L.Mp * 4);
    L.bi_t = L.sc_t + up((size_t)L.G * a.N * 4);
    L.bpart = L.bi_t + up((size_t)L.G * a.N * 4);
    L.total = L.bpart + up((size_t)a.N * ((L.G + 31) / 32) * 4);
    return L;
}

template <bool PACKED, int GK>
int launch_main(const DevCtx& dc, const CUtensorMap& mq, const CUtensorMap& mx, const Params& kp,
                dim3 grid, cudaStream_t s) {
    constexpr int smem = Geo<PACKED>::kSmemBytes;
    static int configured[64] = {0};
    auto kern = mma_kernel<PACKED, GK>;
    if (dc.device >= 0 && dc.device < 64 && !configured[dc.device]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return cuda_fail(e);
        configured[dc.device] = 1;
    }
    kern<<<grid, kThreads, smem, s>>>(mq, mx, kp);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

// prep_kernel as a programmatic dependent of the preceding kernel (it waits
// for it before touching any data).
int launch_prep(unsigned blocks, cudaStream_t s, const float* x, __half* xh, float* xsum,
                float* inv, const float* sc, const float* bi, float* sc_t, float* bi_t,
                float* bpart, float qmax, int M, int N, int K, int gs, int G, int Mp) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kPrepThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, prep_kernel, x, xh, xsum, inv, sc, bi, sc_t, bi_t,
                                       bpart, qmax, M, N, K, gs, G, Mp);
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

}  // namespace prefill

bool prefill_eligible(const DevCtx& dc, const GemvArgs& a) {
    const bool packed = a.fmt == FMT_AFF_PACKED;
    if (a.fmt != FMT_AFF_U8 && !packed) return false;
    if (a.M < launch_option(QG_OPT_PREFILL_MIN_M)) return false;
    if (a.gs < 16) return false;
    if (a.K % (packed ? 32 : 16)) return false;
    if (a.K > (1ll << 30) || a.M > (1ll << 30)) return false;
    if (a.N > 65535ll * prefill::kTileN) return false;
    if ((reinterpret_cast<uintptr_t>(a.w[0]) & 15) || (reinterpret_cast<uintptr_t>(a.x) & 15))
        return false;
    if (dc.max_smem_optin < std::max(prefill::Geo<false>::kSmemBytes, prefill::fold_smem_bytes(false)))
        return false;
    return true;
}

size_t prefill_workspace_bytes(const GemvArgs& a) { return prefill::layout(a).total; }

int prefill_launch(const DevCtx& dc, const GemvArgs& a, void* ws, size_t ws_bytes, cudaStream_t s) {
    using namespace prefill;
    const Layout L = layout(a);
    if (!ws || ws_bytes < L.total) return QG_ERR_WORKSPACE;
    const bool packed = a.fmt == FMT_AFF_PACKED;
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    int rc = encoder(&encode);
    if (rc) return rc;
    uint8_t* w8 = static_cast<uint8_t*>(ws);
    __half* xh = reinterpret_cast<__half*>(w8 + L.xh);
    float* xsum = reinterpret_cast<float*>(w8 + L.xsum);
    float* inv = reinterpret_cast<float*>(w8 + L.inv);

    CUtensorMap mx, mq;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
        const cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
        const cuuint32_t box[2] = {kChunk, kTileT};
        const cuuint32_t es[2] = {1, 1};
        if (encode(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xh, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return QG_ERR_UNSUPPORTED;
    }
    {
        const cuuint64_t kb = packed ? a.K / 2 : a.K;
        const cuuint64_t dims[2] = {kb, (cuuint64_t)a.N};
        const cuuint64_t strides[1] = {kb};
        const cuuint32_t box[2] = {(cuuint32_t)(packed ? kChunk / 2 : kChunk), kTileN};
        const cuuint32_t es[2] = {1, 1};
        if (encode(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.w[0]), dims,
                   strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   packed ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return QG_ERR_UNSUPPORTED;
    }

    float* sc_t = reinterpret_cast<float*>(w8 + L.sc_t);
    float* bi_t = reinterpret_cast<float*>(w8 + L.bi_t);
    float* bpart = reinterpret_cast<float*>(w8 + L.bpart);
    const dim3 grid(L.Mp / kTileT, (unsigned)((a.N + kTileN - 1) / kTileN));
    const long long tiles = ((a.N + 31) / 32) * (long long)((L.G + 31) / 32);
    if (tiles > 0x7FFFFFFFll - L.Mp) return QG_ERR_UNSUPPORTED;
    if (launch_option(QG_OPT_PREFILL_FOLD)) {
        int rc2 = launch_prep((unsigned)(L.Mp + tiles), s, a.x, xh, nullptr, inv, a.scales,
                              a.biases, sc_t, bi_t, bpart, packed ? 15.f : 255.f, (int)a.M,
                              (int)a.N, (int)a.K, a.gs, L.G, L.Mp);
        if (rc2 != QG_OK) return rc2;
        FoldParams fp{};
        fp.scales_t = sc_t;
        fp.biases_t = bi_t;
        fp.bpart = bpart;
        fp.GT = (L.G + 31) / 32;
        fp.inv = inv;
        fp.y = a.y[0];
        fp.M = (int)a.M;
        fp.N = (int)a.N;
        fp.K = (int)a.K;
        fp.G = L.G;
        fp.log2gs = __builtin_ctz((unsigned)a.gs);
        fp.err = dc.err;
        return launch_fold_kernel(dc, packed, a.gs == 16, mq, mx, fp, grid, s);
    }
    rc = launch_prep((unsigned)(L.Mp + tiles), s, a.x, xh, xsum, inv, a.scales, a.biases, sc_t,
                     bi_t, nullptr, 0.f, (int)a.M, (int)a.N, (int)a.K, a.gs, L.G, L.Mp);
    if (rc != QG_OK) return rc;

    Params kp{};
    kp.scales_t = sc_t;
    kp.biases_t = bi_t;
    kp.y = a.y[0];
    kp.xsum = xsum;
    kp.inv = inv;
    kp.M = (int)a.M;
    kp.N = (int)a.N;
    kp.K = (int)a.K;
    kp.G = L.G;
    kp.Mp = L.Mp;
    kp.gs = a.gs;
    kp.spgs = a.gs >= 2 * kChunk ? a.gs / (2 * kChunk) : 1;  // steps per group (gs >= 128)
    kp.err = dc.err;
    if (a.gs == 16)
        return packed ? launch_main<true, 1>(dc, mq, mx, kp, grid, s)
                      : launch_main<false, 1>(dc, mq, mx, kp, grid, s);
    if (a.gs == 32)
        return packed ? launch_main<true, 2>(dc, mq, mx, kp, grid, s)
                      : launch_main<false, 2>(dc, mq, mx, kp, grid, s);
    if (a.gs == 64)
        return packed ? launch_main<true, 4>(dc, mq, mx, kp, grid, s)
                      : launch_main<false, 4>(dc, mq, mx, kp, grid, s);
    return packed ? launch_main<true, 8>(dc, mq, mx, kp, grid, s)
                  : launch_main<false, 8>(dc, mq, mx, kp, grid, s);
}

}  // namespace qg
