// The fast GEMV kernel template (16-byte aligned weight rows), included by
// one translation unit per weight format.
//
// Pages: fused_dual_proj_q4_0.rs (mlx-native 0.9.1), q4_k_gemv_v2.rs
// (ferrum-kernels 0.7.7) and qmm_affine.rs (mlx-native 0.21.1) define the
// operations; their Metal kernels are not reused. Design for sm_103a:
//
//  * One persistent CTA per SM: W consumer warps + 1 producer warp. CTAs take
//    contiguous, balanced ranges of row chunks (R consecutive rows of one
//    weight matrix; the dual projection is the row list of W_a then W_b).
//  * The producer lane streams each chunk's bytes (codes, and for the affine
//    format the chunk's scales and biases) from HBM into a ring of shared
//    memory stages with 1-D TMA bulk copies completing on mbarriers, with an
//    evict-first L2 policy. A whole SM's share of the weights can be in flight
//    at once without occupying registers.
//  * x (one k-slice of it) is staged once per CTA in shared memory: permuted so
//    that every lane's inputs for a pass are consecutive float4 (conflict-free)
//    and pre-multiplied by a power of two per element (see below). Per-unit
//    sums of the unscaled x are kept beside it for the formats with an offset
//    term (Q4_K min, affine bias).
//  * Stage ownership: chunk i of a CTA lands in stage i % S, and stage st is
//    always consumed by warp st % W, so every stage's uses are awaited in order.
//  * Lane <-> unit: each lane owns one unit of UE consecutive weights of a row
//    (a Q4_0 block of 32, half a Q4_K super-block of 64 = two sub-blocks, 32
//    affine codes), so per-block scales are read once per 32/64 weights. A warp
//    covers a pass of 32 units and walks the R rows of its chunk.
//  * Decode: a nibble at bit 4p of a 32-bit word becomes the exact float
//    2^23 + q * 2^(4p) with one LOP3 ((word & mask) | 0x4B000000) for bit
//    positions up to 19; the three nibbles above bit 19 use the word shifted
//    right by 12. One packed f32x2 subtraction of (2^23 + bias * 2^(4p)) leaves
//    2^(4p) * (q - bias) exactly. The matching x was pre-multiplied by
//    2^-(4p), so each product equals (q - bias) * x exactly before its single
//    rounding in the packed f32x2 FMA (exact for |x| >= 2^-110; smaller
//    magnitudes could lose bits to subnormal rounding). Bytes (one affine code
//    per byte) go through PRMT into 2^23 + q with no scaling.
//  * Partial sums of the R*M outputs are reduced across the warp with a
//    transposing butterfly and written once.
//
// Every output's arithmetic depends only on (format, M bucket, K slicing),
// never on the CTA, warp, chunk size or matrix that produced it: the dual
// projection is bitwise equal to two single projections, and packed affine
// codes give bitwise the same y as one code per byte.
#pragma once

#include <cuda_fp16.h>

#include "qg_internal.cuh"

namespace qg {
namespace fast {

// ------------------------------------------------------------ format traits
template <int FMT> struct Fmt;

template <> struct Fmt<FMT_Q4_0> {
    static constexpr int UE = 32;            // weights per lane unit (one block)
    static constexpr int WORDS = 4;          // 8-weight words per unit
    static constexpr int UNIT_BYTES = 18;
    static constexpr bool kSums = false;
    static constexpr int NH = 1;
    static constexpr float kBias = 8.0f;
};
template <> struct Fmt<FMT_Q4_K> {
    static constexpr int UE = 64;            // one 32-byte nibble chunk: sub-blocks 2c, 2c+1
    static constexpr int WORDS = 8;
    static constexpr int UNIT_BYTES = 36;    // 144 bytes per 4 units
    static constexpr bool kSums = true;
    static constexpr int NH = 2;
    static constexpr float kBias = 0.0f;
};
template <> struct Fmt<FMT_AFF_U8> {
    static constexpr int UE = 32;
    static constexpr int WORDS = 4;
    static constexpr int UNIT_BYTES = 32;
    static constexpr bool kSums = true;
    static constexpr int NH = 1;
    static constexpr float kBias = 0.0f;
};
template <> struct Fmt<FMT_AFF_PACKED> {
    static constexpr int UE = 32;
    static constexpr int WORDS = 4;
    static constexpr int UNIT_BYTES = 16;
    static constexpr bool kSums = true;
    static constexpr int NH = 1;
    static constexpr float kBias = 0.0f;
};

// log2 of the scale 2^s carried by the decoded value of element j of a unit
// (and removed from x at staging time).
template <int FMT>
__host__ __device__ __forceinline__ int elem_shift(int j) {
    if (FMT == FMT_AFF_U8) return 0;
    if (FMT == FMT_AFF_PACKED) {
        const int e = j & 7;  // nibble e of the word holding elements 8w..8w+7
        return e <= 4 ? 4 * e : 4 * (e - 3);
    }
    // Q4_0 (32 = 16 low + 16 high) and Q4_K (64 = 32 low + 32 high): byte t of
    // a word holds a low-half element in bits 8t..8t+3 and a high-half element
    // in bits 8t+4..8t+7.
    const int half = (FMT == FMT_Q4_0) ? 16 : 32;
    const int t = j & 3;
    const int p = 2 * t + (j >= half ? 1 : 0);  // nibble position in the word
    return p <= 4 ? 4 * p : 4 * (p - 3);
}

// Programmatic dependent launch: let the next kernel on the stream launch /
// wait until the preceding kernel's memory operations are visible. Both are
// no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Per-kernel parameters (by value).
struct Params {
    const uint8_t* w[2];
    float* out[2];
    float* partial;
    const float* x;
    const float* s;
    const float* b;
    int M, N, K;
    int log2gs;
    int nw;
    int klen, P, units;        // k-slice length, passes, units per row slice
    int chunks_per_w, total_chunks;
    int chunk_base, chunk_rem;  // total_chunks = chunk_base * gridDim.x + chunk_rem
    int ahead;                  // chunks in flight at most (0: up to S)
    int S, stage_bytes;
    int q_stride, sb_stride, sb_off;
    long long q_row_bytes;
    int G;
    int KS;
    int xs_bytes, xsum_bytes;
    uint32_t magic;            // 0x4B000000, passed in so it stays in a register
    unsigned* err;
    int dep_wait;              // 1: wait for the preceding kernel before reading x / writing y
};

// 2^23 + bias * 2^s as the constant removed by the packed subtraction.
__device__ __forceinline__ float magic_sub(float bias, int s) {
    return 8388608.0f + bias * (float)(1 << s);
}

// (v & MASK) | mg in one LOP3 (mg arrives in a register so that the mask can
// be the instruction's immediate).
template <uint32_t MASK>
__device__ __forceinline__ float and_or(uint32_t v, uint32_t mg) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(v), "n"(MASK), "r"(mg));
    return __uint_as_float(d);
}

// Four packed pairs of exact values 2^s * (q - bias) from one word of eight
// nibbles; pair order matches x chunks A (.xy, .zw) then B (.xy, .zw).
// mg = 0x4B000000 (the exponent of 2^23); c[i] = the four constant pairs.
template <int FMT>
__device__ __forceinline__ void decode_nibbles(uint32_t v, uint32_t mg, const float2 (&c)[4],
                                               float2 (&f)[4]) {
    const uint32_t v2 = v >> 12;
    const float n0 = and_or<0x0000Fu>(v, mg);   // nibble 0, 2^0
    const float n1 = and_or<0x000F0u>(v, mg);   // nibble 1, 2^4
    const float n2 = and_or<0x00F00u>(v, mg);   // nibble 2, 2^8
    const float n3 = and_or<0x0F000u>(v, mg);   // nibble 3, 2^12
    const float n4 = and_or<0xF0000u>(v, mg);   // nibble 4, 2^16
    const float n5 = and_or<0x00F00u>(v2, mg);  // nibble 5, 2^8
    const float n6 = and_or<0x0F000u>(v2, mg);  // nibble 6, 2^12
    const float n7 = and_or<0xF0000u>(v2, mg);  // nibble 7, 2^16
    if (FMT == FMT_AFF_PACKED) {
        // element e = nibble e: pairs (0,1) (2,3) (4,5) (6,7)
        f[0] = __fadd2_rn(make_float2(n0, n1), c[0]);
        f[1] = __fadd2_rn(make_float2(n2, n3), c[1]);
        f[2] = __fadd2_rn(make_float2(n4, n5), c[2]);
        f[3] = __fadd2_rn(make_float2(n6, n7), c[3]);
    } else {
        // low-half elements t = 0..3 are nibbles 0,2,4,6; high-half 1,3,5,7
        f[0] = __fadd2_rn(make_float2(n0, n2), c[0]);
        f[1] = __fadd2_rn(make_float2(n4, n6), c[1]);
        f[2] = __fadd2_rn(make_float2(n1, n3), c[2]);
        f[3] = __fadd2_rn(make_float2(n5, n7), c[3]);
    }
}

// The constant pairs -(2^23 + bias * 2^s) matching decode_nibbles' pairs.
template <int FMT>
__device__ __forceinline__ void decode_consts(float2 (&c)[4]) {
    const float b = Fmt<FMT>::kBias;
    if (FMT == FMT_AFF_PACKED) {
        c[0] = make_float2(-magic_sub(b, 0), -magic_sub(b, 4));
        c[1] = make_float2(-magic_sub(b, 8), -magic_sub(b, 12));
        c[2] = make_float2(-magic_sub(b, 16), -magic_sub(b, 8));
        c[3] = make_float2(-magic_sub(b, 12), -magic_sub(b, 16));
    } else {
        c[0] = make_float2(-magic_sub(b, 0), -magic_sub(b, 8));
        c[1] = make_float2(-magic_sub(b, 16), -magic_sub(b, 12));
        c[2] = make_float2(-magic_sub(b, 4), -magic_sub(b, 12));
        c[3] = make_float2(-magic_sub(b, 8), -magic_sub(b, 16));
    }
}

// Eight bytes (two words) -> four pairs of exact code values, element order.
__device__ __forceinline__ void decode_bytes(uint32_t v0, uint32_t v1, uint32_t MG, float2 (&f)[4]) {
    const float2 c = make_float2(-8388608.0f, -8388608.0f);
    f[0] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(v0, MG, 0x7540)),
                                  __uint_as_float(__byte_perm(v0, MG, 0x7541))), c);
    f[1] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(v0, MG, 0x7542)),
                                  __uint_as_float(__byte_perm(v0, MG, 0x7543))), c);
    f[2] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(v1, MG, 0x7540)),
                                  __uint_as_float(__byte_perm(v1, MG, 0x7541))), c);
    f[3] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(v1, MG, 0x7542)),
                                  __uint_as_float(__byte_perm(v1, MG, 0x7543))), c);
}

// s += f . (xa, xb) as four packed FMAs in a fixed order.
__device__ __forceinline__ float2 dot8(const float2 (&f)[4], const float4& xa, const float4& xb,
                                       float2 s) {
    s = __ffma2_rn(f[0], make_float2(xa.x, xa.y), s);
    s = __ffma2_rn(f[1], make_float2(xa.z, xa.w), s);
    s = __ffma2_rn(f[2], make_float2(xb.x, xb.y), s);
    s = __ffma2_rn(f[3], make_float2(xb.z, xb.w), s);
    return s;
}

// Which x chunks (of 4 elements within the lane's unit) word w pairs with.
template <int FMT>
__device__ __forceinline__ int chunk_a(int w) {
    return (FMT == FMT_AFF_U8 || FMT == FMT_AFF_PACKED) ? 2 * w : w;
}
template <int FMT>
__device__ __forceinline__ int chunk_b(int w) {
    return (FMT == FMT_AFF_U8 || FMT == FMT_AFF_PACKED) ? 2 * w + 1
                                                        : w + Fmt<FMT>::UE / 8;
}

// Q4_K (scale, min) pair of sub-block j from the 12 packed bytes as 3 words.
__device__ __forceinline__ void q4k_pair(uint32_t s0, uint32_t s1, uint32_t s2, int j, int& sc,
                                         int& mn) {
    const int sh = 8 * (j & 3);
    const uint32_t b0 = (s0 >> sh) & 0xFF, b1 = (s1 >> sh) & 0xFF, b2 = (s2 >> sh) & 0xFF;
    if (j < 4) {
        sc = b0 & 63;
        mn = b1 & 63;
    } else {
        sc = (b2 & 15) | ((b0 >> 6) << 4);
        mn = (b2 >> 4) | ((b1 >> 6) << 4);
    }
}

// Per-(row, unit) scale data.
struct UnitScale {
    float a0, m0, a1, m1;  // Q4_0: a0 = d. Q4_K: d*sc and dmin*m of both halves.
};                         // affine: a0 = s, m0 = b.

// Warp reduction of V values at once; lane l ends with value l / (32 / V).
template <int V>
__device__ __forceinline__ void butterfly(float (&v)[V], int lane) {
    int cur = V;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        if (cur > 1) {
            const int half = cur / 2;
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                if (i < half) {
                    const float send = upper ? v[i] : v[i + half];
                    const float keep = upper ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
            cur = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
        }
    }
}

// Eight consumer warps with M bucket 1 leave room for two CTAs per SM (this
// launch's and the next one's); with larger M buckets they run one CTA per SM
// and up to 168 registers a thread (three warps per SM sub-partition).
template <int FMT, int MT, int R, int W, int GW>
__global__ void __launch_bounds__((W + 1) * 32, (W == 8 && MT == 1) ? 2 : 1) gemv_fast_kernel(const Params p) {
    using F = Fmt<FMT>;
    constexpr int UE = F::UE;
    constexpr int NCH = UE / 4;       // float4 chunks of x per unit
    constexpr int PASS = 32 * UE;
    constexpr bool kAffine = (FMT == FMT_AFF_U8 || FMT == FMT_AFF_PACKED);
    constexpr int kThreadsC = W * 32;
    constexpr int SR = R;             // rows per stage (all GW warps of a group share them)
    constexpr int NG = W / GW;        // warp groups
    constexpr int RB = (MT == 1) ? (R < 4 ? R : 4) : (R < 2 ? R : 2);  // row batch

    extern __shared__ __align__(128) uint8_t smem[];
    float* xs = reinterpret_cast<float*>(smem);
    float* xsum = reinterpret_cast<float*>(smem + p.xs_bytes);
    uint8_t* stages = smem + p.xs_bytes + p.xsum_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(stages + (size_t)p.S * p.stage_bytes);
    uint64_t* empty = full + p.S;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ks = blockIdx.y;
    const int k0 = ks * p.klen;
    // CTA b takes chunk_base chunks, plus one more when b < chunk_rem.
    const int c_begin = (int)blockIdx.x * p.chunk_base + min((int)blockIdx.x, p.chunk_rem);
    const int c_end = c_begin + p.chunk_base + ((int)blockIdx.x < p.chunk_rem ? 1 : 0);
    const int n_local = c_end - c_begin;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.S; ++i) {
            mbar_init(smem_addr(&full[i]), 1);
            mbar_init(smem_addr(&empty[i]), GW);
        }
        fence_mbar_init();
        int* c0 = reinterpret_cast<int*>(smem + p.xs_bytes + p.xsum_bytes) - p.S;
        for (int i = 0; i < p.S; ++i) c0[i] = 0;
    }
    __syncthreads();

    // ------------------------------------------------------------ producer
    // Weights, scales and biases are read before griddepcontrol.wait: under
    // programmatic dependent launch they must not be written by the kernel
    // that precedes this one on the stream (the documented contract of that
    // launch mode). Without it the wait is a no-op.
    if (warp == W) {
        if (lane != 0) return;
        const uint64_t pol = l2_evict_first();
        const long long q_off = (long long)k0 / UE * F::UNIT_BYTES;
        const int g_off = kAffine ? (k0 >> p.log2gs) : 0;
        int issued = 0;
        bool ok = true;
        for (int i = 0; i < n_local; ++i) {
            const int st = i % p.S, use = i / p.S;
            if (use > 0 && !mbar_wait(smem_addr(&empty[st]), (use - 1) & 1)) {
                report_error(p.err, DEVERR_WAIT_EMPTY);
                ok = false;
                break;
            }
            // At most `ahead` chunks in flight: chunk i is requested once chunk
            // i - ahead has landed, so that every SM's first chunks are not
            // queued behind the whole grid's traffic (ahead <= S, so the
            // awaited phase is the latest one of that stage).
            if (p.ahead > 0 && i >= p.ahead) {
                const int j = i - p.ahead;
                if (!mbar_wait(smem_addr(&full[j % p.S]), (j / p.S) & 1)) {
                    report_error(p.err, DEVERR_WAIT_FULL);
                    ok = false;
                    break;
                }
            }
            const int cid = c_begin + i;
            const int wi = cid / p.chunks_per_w;
            const int row0 = (cid - wi * p.chunks_per_w) * SR;
            const int rows = min(SR, p.N - row0);
            uint8_t* dst = stages + (size_t)st * p.stage_bytes;
            const uint32_t bar = smem_addr(&full[st]);
            uint32_t bytes = (uint32_t)(rows * p.q_stride);
            if (kAffine) bytes += 2u * rows * p.sb_stride;
            mbar_arrive_expect_tx(bar, bytes);
            const uint8_t* wsrc = p.w[wi] + (long long)row0 * p.q_row_bytes + q_off;
            if (p.KS == 1) {
                bulk_g2s(smem_addr(dst), wsrc, rows * p.q_stride, bar, pol);
                if (kAffine) {
                    bulk_g2s(smem_addr(dst + p.sb_off), p.s + (long long)row0 * p.G,
                             rows * p.sb_stride, bar, pol);
                    bulk_g2s(smem_addr(dst + p.sb_off + SR * p.sb_stride),
                             p.b + (long long)row0 * p.G, rows * p.sb_stride, bar, pol);
                }
            } else {
                for (int r = 0; r < rows; ++r) {
                    bulk_g2s(smem_addr(dst + r * p.q_stride), wsrc + r * p.q_row_bytes,
                             p.q_stride, bar, pol);
                    if (kAffine) {
                        const long long go = (long long)(row0 + r) * p.G + g_off;
                        bulk_g2s(smem_addr(dst + p.sb_off + r * p.sb_stride), p.s + go,
                                 p.sb_stride, bar, pol);
                        bulk_g2s(smem_addr(dst + p.sb_off + (SR + r) * p.sb_stride), p.b + go,
                                 p.sb_stride, bar, pol);
                    }
                }
            }
            issued = i + 1;
            // Once the first stages are on their way, the next kernel in the
            // stream may start its own prologue.
            if (i == min(n_local, p.S) - 1) pdl_launch_dependents();
        }
        if (n_local == 0) pdl_launch_dependents();
        if (!ok) {
            // Let every stage's latest copies land before shared memory is released.
            for (int st = 0; st < p.S && st < issued; ++st) {
                const int last = st + ((issued - 1 - st) / p.S) * p.S;
                if (!mbar_wait(smem_addr(&full[st]), (last / p.S) & 1))
                    report_error(p.err, DEVERR_WAIT_DRAIN);
            }
        }
        return;
    }

    // x and y may be produced / consumed by the preceding kernel (unless the
    // caller declared the calls independent and no split-K workspace is in
    // use).
    if (p.dep_wait) pdl_wait();

    // ------------------------------------------------- stage x (consumers)
    // Shift-only index math: UE and PASS are powers of two. Every thread
    // issues 16 float4 loads (over all MT rows) before its first store, so the
    // prologue costs about one L2 round trip for the common shapes.
    constexpr int LOG_UE = (UE == 64) ? 6 : 5;
    constexpr int LOG_PASS = LOG_UE + 5;
    {
        const int span = p.P * PASS;
        const int quads = span >> 2;
        const bool vec = ((reinterpret_cast<uintptr_t>(p.x) & 15) == 0) && ((p.K & 3) == 0);
        // Quads per thread per round, for each of the MT rows: at most 16
        // loads in flight, and no more rounds than the slice needs.
        constexpr int QU = 16 / MT;
        const int per_thread = (quads + kThreadsC - 1) / kThreadsC;
#pragma unroll 1
        for (int u0 = 0; u0 < per_thread; u0 += QU) {
            float4 v[QU][MT];
#pragma unroll
            for (int u = 0; u < QU; ++u) {
                const int e = (threadIdx.x + (u0 + u) * kThreadsC) << 2;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    v[u][m] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (u0 + u < per_thread && m < p.M && e < p.klen) {
                        const float* src = p.x + (long long)m * p.K + k0 + e;
                        if (vec) {
                            v[u][m] = *reinterpret_cast<const float4*>(src);
                        } else {
                            v[u][m].x = src[0];
                            v[u][m].y = src[1];
                            v[u][m].z = src[2];
                            v[u][m].w = src[3];
                        }
                    }
                }
                if (u0 + u + 1 >= per_thread) break;
            }
#pragma unroll
            for (int u = 0; u < QU; ++u) {
                if (u0 + u >= per_thread) break;
                const int e = (threadIdx.x + (u0 + u) * kThreadsC) << 2;
                if (e >= span) break;
                const int pp = e >> LOG_PASS, within = e & (PASS - 1);
                const int ln = within >> LOG_UE, j = within & (UE - 1);
                const float s0 = __uint_as_float((uint32_t)(127 - elem_shift<FMT>(j)) << 23);
                const float s1 = __uint_as_float((uint32_t)(127 - elem_shift<FMT>(j + 1)) << 23);
                const float s2 = __uint_as_float((uint32_t)(127 - elem_shift<FMT>(j + 2)) << 23);
                const float s3 = __uint_as_float((uint32_t)(127 - elem_shift<FMT>(j + 3)) << 23);
                const int off = ((pp * NCH + (j >> 2)) * 32 + ln) * 4;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float4 o = make_float4(v[u][m].x * s0, v[u][m].y * s1, v[u][m].z * s2,
                                                 v[u][m].w * s3);
                    *reinterpret_cast<float4*>(xs + m * span + off) = o;
                }
            }
        }
        if (F::kSums) {
            // Sums of the unscaled x over each unit half, in natural element
            // order, read back from the staged copy (the power-of-two scaling
            // is undone exactly).
            named_bar_sync(1, kThreadsC);
            constexpr int HL = UE / F::NH;  // elements per summed half
            const int per_m = p.P * 32 * F::NH;
            for (int idx = threadIdx.x; idx < MT * per_m; idx += kThreadsC) {
                const int m = idx / per_m, r = idx - m * per_m;  // r = (pp * 32 + lane) * NH + h
                const int h = r % F::NH, ln = (r / F::NH) & 31, pp = r / (F::NH * 32);
                const float* xsrc = xs + m * span;
                float sacc = 0.0f;
#pragma unroll 8
                for (int jj = 0; jj < HL; ++jj) {
                    const int j = h * HL + jj;
                    const float v = xsrc[((pp * NCH + (j >> 2)) * 32 + ln) * 4 + (j & 3)];
                    sacc += v * __uint_as_float((uint32_t)(127 + elem_shift<FMT>(j)) << 23);
                }
                xsum[idx] = sacc;
            }
        }
    }
    named_bar_sync(1, kThreadsC);

    const float4* xs4 = reinterpret_cast<const float4*>(xs);
    const uint32_t mg = p.magic;
    float2 cst[4];
    if (FMT != FMT_AFF_U8) decode_consts<FMT>(cst);
    // Cross-warp partial sums of a stage, [S][GW][V], and per-stage arrival
    // counters, [S], kept at the end of the x-sum region (see the planner).
    constexpr int V = MT * R;
    int* cnt = reinterpret_cast<int*>(xsum + (p.xsum_bytes >> 2)) - p.S;
    float* red = reinterpret_cast<float*>(cnt) - p.S * GW * V;

    // Stage st is consumed only by warp group st % NG (see the file comment):
    // with S a multiple of NG group g takes stages g, g+NG, ...; with S < NG,
    // group g < S takes g, g+S, ... The GW warps of a group split the passes
    // of the k-slice (warp gw takes passes gw, gw+GW, ...) for all R rows of
    // the stage and add their partial sums in warp order.
    const int grp = warp / GW, gw = warp - grp * GW;
    const int stride = (p.S >= NG) ? NG : p.S;
    int st = grp, use = 0;
    // After a wait gives up the warp keeps stepping through its stages (and
    // the group's named barriers) without computing, so that no other warp
    // of the group is left waiting at a barrier.
    bool dead = false;
    for (int i = grp; i < n_local && grp < stride; i += stride) {
        if (!dead && !mbar_wait(smem_addr(&full[st]), use & 1)) {
            report_error(p.err, DEVERR_WAIT_FULL);
            dead = true;
        }
        const int cid = c_begin + i;
        const int wi = cid / p.chunks_per_w;
        const int row0 = (cid - wi * p.chunks_per_w) * R;
        const int rows = min(R, p.N - row0);
        const uint8_t* stg = stages + (size_t)st * p.stage_bytes;
        // Rows past the end of a matrix (ragged last stage) are computed from
        // stale stage bytes and never written.

        float acc[MT][R];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < R; ++r) acc[m][r] = 0.0f;

#pragma unroll 1
        for (int pp = gw; pp < (dead ? 0 : p.P); pp += GW) {
            const int u = pp * 32 + lane;           // unit index within the row slice
            const bool valid = u < p.units;
            const int uc = valid ? u : 0;           // clamp for address math
            const int ub = uc * F::UNIT_BYTES;      // unit's byte offset in a row
            const float4* xp = xs4 + pp * NCH * 32 + lane;
            // Byte offset of the unit's nibble words inside a row (Q4_K, affine).
            const int qo = (FMT == FMT_Q4_K) ? (uc >> 2) * 144 + 16 + 32 * (uc & 3) : ub;
            const uint32_t qsh = 16u + (uint32_t)(ub & 2) * 8u;  // Q4_0: 16 or 32

            // Unscaled x sums of the lane's unit halves, per input row.
            float sx0[MT], sx1[MT];
            if (F::kSums) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float* xsp = xsum + ((m * p.P + pp) * 32 + lane) * F::NH;
                    sx0[m] = xsp[0];
                    sx1[m] = (F::NH > 1) ? xsp[F::NH - 1] : 0.0f;
                }
            }

            // Rows in batches of RB: the batch's block windows / unit scales stay
            // in registers while each x word is loaded once and used RB times.
#pragma unroll
            for (int rb0 = 0; rb0 < R; rb0 += RB) {
                UnitScale us[RB];
                uint32_t win[RB][5];
#pragma unroll
                for (int b = 0; b < RB; ++b) {
                    const int r = rb0 + b;
                    const uint8_t* rowr = stg + r * p.q_stride;
                    if (FMT == FMT_Q4_0) {
                        const uint32_t* wp = reinterpret_cast<const uint32_t*>(rowr + (ub & ~3));
#pragma unroll
                        for (int q = 0; q < 5; ++q) win[b][q] = wp[q];
                        const uint32_t dbits =
                            __funnelshift_r(win[b][0], win[b][1], qsh - 16u) & 0xFFFFu;
                        us[b].a0 = __half2float(__ushort_as_half((unsigned short)dbits));
                    } else if (FMT == FMT_Q4_K) {
                        const int c = uc & 3;
                        const uint4 h = *reinterpret_cast<const uint4*>(rowr + (uc >> 2) * 144);
                        int sc0, mn0, sc1, mn1;
                        q4k_pair(h.y, h.z, h.w, 2 * c, sc0, mn0);
                        q4k_pair(h.y, h.z, h.w, 2 * c + 1, sc1, mn1);
                        const float d =
                            __half2float(__ushort_as_half((unsigned short)(h.x & 0xFFFF)));
                        const float dm = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
                        us[b].a0 = d * (float)sc0;
                        us[b].m0 = dm * (float)mn0;
                        us[b].a1 = d * (float)sc1;
                        us[b].m1 = dm * (float)mn1;
                    } else {
                        const int g = (uc * UE) >> p.log2gs;
                        us[b].a0 =
                            reinterpret_cast<const float*>(stg + p.sb_off + r * p.sb_stride)[g];
                        us[b].m0 =
                            reinterpret_cast<const float*>(stg + p.sb_off + (R + r) * p.sb_stride)[g];
                    }
                }

                // Packed partial sums per (m, row); Q4_K keeps its two halves apart.
                float2 s_lo[MT][RB], s_hi[MT][RB];
#pragma unroll
                for (int m = 0; m < MT; ++m)
#pragma unroll
                    for (int b = 0; b < RB; ++b) {
                        s_lo[m][b] = make_float2(0.0f, 0.0f);
                        s_hi[m][b] = make_float2(0.0f, 0.0f);
                    }
#pragma unroll
                for (int w = 0; w < F::WORDS; ++w) {
                    // Decode the word of every row of the batch once, then stream x
                    // row by row (only one x row's chunks live at a time; the
                    // per-output arithmetic order is the same as x-major order).
                    float2 f[RB][4];
#pragma unroll
                    for (int b = 0; b < RB; ++b) {
                        const uint8_t* rowr = stg + (rb0 + b) * p.q_stride;
                        if (FMT == FMT_Q4_0) {
                            decode_nibbles<FMT>(__funnelshift_rc(win[b][w], win[b][w + 1], qsh), mg,
                                                cst, f[b]);
                        } else if (FMT == FMT_Q4_K || FMT == FMT_AFF_PACKED) {
                            const uint32_t v =
                                *reinterpret_cast<const uint32_t*>(rowr + qo + 4 * w);
                            decode_nibbles<FMT>(v, mg, cst, f[b]);
                        } else {
                            const uint2 v = *reinterpret_cast<const uint2*>(rowr + qo + 8 * w);
                            decode_bytes(v.x, v.y, mg, f[b]);
                        }
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const float4 xa = xp[(m * p.P * NCH + chunk_a<FMT>(w)) * 32];
                        const float4 xb = xp[(m * p.P * NCH + chunk_b<FMT>(w)) * 32];
#pragma unroll
                        for (int b = 0; b < RB; ++b) {
                            if (FMT == FMT_Q4_K) {
                                s_lo[m][b] = __ffma2_rn(f[b][0], make_float2(xa.x, xa.y), s_lo[m][b]);
                                s_lo[m][b] = __ffma2_rn(f[b][1], make_float2(xa.z, xa.w), s_lo[m][b]);
                                s_hi[m][b] = __ffma2_rn(f[b][2], make_float2(xb.x, xb.y), s_hi[m][b]);
                                s_hi[m][b] = __ffma2_rn(f[b][3], make_float2(xb.z, xb.w), s_hi[m][b]);
                            } else {
                                s_lo[m][b] = dot8(f[b], xa, xb, s_lo[m][b]);
                            }
                        }
                    }
                }
                // Apply the unit scales once per (row, unit); invalid lanes add 0.
#pragma unroll
                for (int b = 0; b < RB; ++b) {
                    const int r = rb0 + b;
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        float a = acc[m][r];
                        if (FMT == FMT_Q4_0) {
                            a = __fmaf_rn(us[b].a0, s_lo[m][b].x + s_lo[m][b].y, a);
                        } else if (FMT == FMT_Q4_K) {
                            a = __fmaf_rn(us[b].a0, s_lo[m][b].x + s_lo[m][b].y, a);
                            a = __fmaf_rn(-us[b].m0, sx0[m], a);
                            a = __fmaf_rn(us[b].a1, s_hi[m][b].x + s_hi[m][b].y, a);
                            a = __fmaf_rn(-us[b].m1, sx1[m], a);
                        } else {
                            a = __fmaf_rn(us[b].a0, s_lo[m][b].x + s_lo[m][b].y, a);
                            a = __fmaf_rn(us[b].m0, sx0[m], a);
                        }
                        acc[m][r] = valid ? a : acc[m][r];
                    }
                }
            }
        }
        float vals[V];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < R; ++r) vals[m * R + r] = acc[m][r];
        butterfly<V>(vals, lane);
        constexpr int kSpan = 32 / V;
        const bool holder = (lane % kSpan) == 0;
        const int v = lane / kSpan;
        float total = vals[0];
        bool writer = true;
        if (GW > 1) {
            // The last warp of the group to finish this stage adds the GW
            // partial sums in warp order; the others move on without waiting.
            float* rs = red + (size_t)st * GW * V;
            if (holder) rs[gw * V + v] = total;
            __threadfence_block();
            __syncwarp();
            int last = 0;
            if (lane == 0) last = (atomicAdd(&cnt[st], 1) == GW - 1);
            last = __shfl_sync(0xffffffffu, last, 0);
            writer = last != 0;
            if (writer) {
                __threadfence_block();
                total = rs[v];
#pragma unroll
                for (int g2 = 1; g2 < GW; ++g2) total += rs[g2 * V + v];
                __syncwarp();
                if (lane == 0) cnt[st] = 0;
            }
        }
        if (writer && holder) {
            const int m = v / R, r = v % R;
            if (m < p.M && r < rows) {
                const long long o = (long long)m * p.N + row0 + r;
                if (p.KS == 1)
                    p.out[wi][o] = total;
                else
                    p.partial[((long long)(ks * p.nw + wi) * p.M) * p.N + o] = total;
            }
        }
        // The stage (and its partial-sum slot) is released only after this
        // warp is done with both.
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[st]));
        st += stride;
        if (st >= p.S) {
            st -= p.S;
            ++use;
        }
    }
}

// Launch helper used by the per-format translation units. With pdl set the
// kernel is launched with programmatic stream serialization, so that it can
// start (and stream its weights) while the previous kernel drains.
template <int FMT, int MT, int R, int W, int GW>
int launch(const DevCtx& dc, const Params& kp, int grid_x, int smem, bool pdl, cudaStream_t s) {
    auto kern = gemv_fast_kernel<FMT, MT, R, W, GW>;
    static int configured[64] = {0};
    if (dc.device >= 0 && dc.device < 64 && configured[dc.device] < smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             dc.max_smem_optin);
        if (e != cudaSuccess) return cuda_fail(e);
        configured[dc.device] = dc.max_smem_optin;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, kp.KS);
    cfg.blockDim = dim3((W + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, kp);
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

}  // namespace fast
}  // namespace qg

namespace qg {
namespace fast {

// Largest rows-per-stage per (format, M bucket, consumer warps) that compiles
// without register spills. An SM sub-partition holds 16 K registers, so the
// warps it runs share them: 16 consumer warps + producer (five on one
// sub-partition) cap a thread at 96 registers, 12 + producer (four) at 128,
// and 8 + producer (three) at 168 when one CTA runs per SM. Q4_K with M
// bucket 8 runs 8 consumer warps to take two rows per stage.
__host__ __device__ constexpr int max_rows(int fmt, int MT, int W) {
    return fmt == FMT_Q4_0   ? (MT == 1 ? 16 : MT == 8 ? 2 : 4)
           : fmt == FMT_Q4_K ? (MT == 1 ? 4 : MT == 8 ? (W == 8 ? 2 : 1) : 2)
                             : (MT == 1 ? 16 : 2);
}

// (MT, R, GW) -> kernel instantiation: R rows per stage, shared by a group of
// GW warps that split the passes. MT <= 2 runs 16 consumer warps, larger M 12.
template <int FMT, int MT, int W, int R>
int dispatch_gw(const DevCtx& dc, const Params& kp, int GW, int grid, int smem, bool pdl,
                cudaStream_t s) {
    if constexpr (R > max_rows(FMT, MT, W)) {
        return QG_ERR_UNSUPPORTED;
    } else {
        switch (GW) {
            case 1: return launch<FMT, MT, R, W, 1>(dc, kp, grid, smem, pdl, s);
            case 2: return launch<FMT, MT, R, W, 2>(dc, kp, grid, smem, pdl, s);
            default: return launch<FMT, MT, R, W, 4>(dc, kp, grid, smem, pdl, s);
        }
    }
}

template <int FMT>
int dispatch(const DevCtx& dc, const Params& kp, int MT, int R, int GW, int W, int grid,
             int smem, bool pdl, cudaStream_t s) {
    if (MT == 1 && W == 8) {
        // Eight consumer warps and at most 113 registers: two CTAs (this launch's
        // and the next one's) fit on an SM.
        if (R <= 4) return dispatch_gw<FMT, 1, 8, 4>(dc, kp, GW, grid, smem, pdl, s);
        if (R == 8) return dispatch_gw<FMT, 1, 8, 8>(dc, kp, GW, grid, smem, pdl, s);
        return dispatch_gw<FMT, 1, 8, 16>(dc, kp, GW, grid, smem, pdl, s);
    }
    switch (MT) {
        case 1:
            if (R <= 2) return dispatch_gw<FMT, 1, 16, 2>(dc, kp, GW, grid, smem, pdl, s);
            if (R == 4) return dispatch_gw<FMT, 1, 16, 4>(dc, kp, GW, grid, smem, pdl, s);
            if (R == 8) return dispatch_gw<FMT, 1, 16, 8>(dc, kp, GW, grid, smem, pdl, s);
            return dispatch_gw<FMT, 1, 16, 16>(dc, kp, GW, grid, smem, pdl, s);
        case 2:
            if (R <= 2) return dispatch_gw<FMT, 2, 16, 2>(dc, kp, GW, grid, smem, pdl, s);
            return dispatch_gw<FMT, 2, 16, 4>(dc, kp, GW, grid, smem, pdl, s);
        case 4:
            if (R <= 2) return dispatch_gw<FMT, 4, 12, 2>(dc, kp, GW, grid, smem, pdl, s);
            return dispatch_gw<FMT, 4, 12, 4>(dc, kp, GW, grid, smem, pdl, s);
        default:
            if constexpr (FMT == FMT_Q4_K) {
                if (W == 8) {
                    if (R <= 1) return dispatch_gw<FMT, 8, 8, 1>(dc, kp, GW, grid, smem, pdl, s);
                    return dispatch_gw<FMT, 8, 8, 2>(dc, kp, GW, grid, smem, pdl, s);
                }
            }
            if (R <= 1) return dispatch_gw<FMT, 8, 12, 1>(dc, kp, GW, grid, smem, pdl, s);
            if (R == 2) return dispatch_gw<FMT, 8, 12, 2>(dc, kp, GW, grid, smem, pdl, s);
            return dispatch_gw<FMT, 8, 12, 4>(dc, kp, GW, grid, smem, pdl, s);
    }
}

}  // namespace fast
}  // namespace qg
