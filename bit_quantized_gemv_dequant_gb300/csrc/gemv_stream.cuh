// The streaming GEMV kernel for M <= 2 (the decode case), included by one
// translation unit per weight format.
//
// Pages: fused_dual_proj_q4_0.rs (mlx-native 0.9.1), q4_k_gemv_v2.rs
// (ferrum-kernels 0.7.7) and qmm_affine.rs (mlx-native 0.21.1) define the
// operations; their Metal kernels are not reused. Design for sm_103a:
//
//  * Work unit: 256 consecutive weights of one row (8 Q4_0 blocks = 144 bytes,
//    one Q4_K super-block = 144 bytes, 256 affine codes = 256 or 128 bytes).
//    A warp step is 32 units, one per lane: RW = 32 / LPR rows of LPR lanes,
//    where LPR (lanes per row) is the largest power of two <= 32 dividing
//    K / 256. A task is RW rows; a lane accumulates its units of the task's
//    row over the task's K / (256 * LPR) steps, and the LPR lanes of a row
//    add their sums with an xor butterfly. The summation order of every
//    output therefore depends only on the format, the M bucket and K: the
//    dual projection is bitwise equal to two single projections.
//  * Weight streaming: each CTA asks L2 to prefetch its contiguous share of
//    the weights at the start. Every warp moves its steps through a private
//    ring of S shared-memory slots with coalesced 16-byte cp.async copies
//    (lane l copies bytes 16 * (l + 32 i) of the step) and reads its own unit
//    back with 16-byte shared loads (the 144-byte lane stride is bank-conflict
//    free). No producer warp, no mbarrier and no spin-wait: cp.async groups
//    complete by themselves.
//  * Programmatic dependent launch: the prefetch is issued before
//    griddepcontrol.wait (weights must not be written by the preceding
//    kernel) and launch_dependents is signalled at once; x is staged after the
//    wait and the ring is filled after x, so that x's loads do not queue
//    behind it. Two CTAs of a launch share an SM when their shared memory fits.
//  * x is staged once per CTA in natural order, one float4 of padding per unit
//    (conflict-free reads of 8 consecutive units), multiplied by 2^c_m with
//    c_m = 119 - floor(log2 max|x_m|) per input row, clamped to [0, 127].
//  * Exact decode without a magic offset: a nibble at bits 4p..4p+3 (p <= 4)
//    of a 32-bit word, masked in place, is the subnormal float q * 2^(4p-149)
//    exactly; the three nibbles above bit 19 are masked out of the word
//    shifted right by 12. A byte code is moved to bits 0..7 with one PRMT.
//    Each packed f32x2 FMA then forms q * x * 2^(c_m - 149 + s) exactly before
//    its single rounding. Q4_0's offset 8 is removed by one exact packed
//    subtraction of 8 * 2^(s-149) first. Every float2 chain component carries
//    one fixed shift s; after 32 weights the four chains are multiplied by
//    their exact 2^-s and added (packed codes: shifts 0..16; byte codes: 0, so
//    both storages add the same values in the same order and give bitwise the
//    same y, barring products in the subnormal range).
//  * The 32-weight scale (Q4_0 d, Q4_K d*sc, affine s) multiplies the chain
//    total into a scaled accumulator; the offset terms (Q4_K dmin*m, affine b)
//    multiply raw per-32 x sums into a second, natural-units accumulator. The
//    scaled one is brought back by 2^(149 - c_m) (exact) before the two are
//    added and the lanes reduced.
#pragma once

#include <cuda_fp16.h>

#include "qg_internal.cuh"

namespace qg {
namespace stream {

// ------------------------------------------------------------ format traits
template <int FMT> struct Fmt;
template <> struct Fmt<FMT_Q4_0> {
    static constexpr int UB = 144;           // bytes per unit of 256 weights
    static constexpr bool kSums = false;
};
template <> struct Fmt<FMT_Q4_K> {
    static constexpr int UB = 144;
    static constexpr bool kSums = true;
};
template <> struct Fmt<FMT_AFF_U8> {
    static constexpr int UB = 256;
    static constexpr bool kSums = true;
};
template <> struct Fmt<FMT_AFF_PACKED> {
    static constexpr int UB = 128;
    static constexpr bool kSums = true;
};

// Per-kernel parameters (by value).
struct Params {
    const uint8_t* w[2];
    float* out[2];
    const float* x;
    const float* s;          // affine scales [N][G]
    const float* b;          // affine biases [N][G]
    int M, N, K;
    int nw;                  // 1, or 2 for the fused dual projection
    int tpr;                 // steps per task = K / (256 * LPR)
    uint32_t tpr_magic;      // tpr > 1: ceil(2^32 / tpr), so r / tpr == __umulhi(r, tpr_magic) for r * tpr < 2^32
    int tasks_per_w;         // ceil(N / RW)
    int total_tasks;         // nw * tasks_per_w
    int tasks_base, tasks_rem;  // total_tasks = tasks_base * gridDim.x + tasks_rem
    int S;                   // ring slots per warp
    int slot_bytes;          // 32 units of codes, then affine s and b
    int sbl;                 // affine: bytes of s (and of b) per lane in a slot
    int log2gs;
    int G;                   // affine groups per row = K / gs
    long long row_bytes;
    int xs_bytes, xsum_bytes;
    uint32_t zero;           // 0, passed at run time (see make_pairk)
};

// ------------------------------------------------------------- PTX helpers
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until at most n of this thread's most recent groups are pending.
__device__ __forceinline__ void cp_wait(int n) {
    switch (n) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
        case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
        case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
        case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    }
}

// Hint L2 to fetch [p, p + bytes); p and bytes multiples of 16.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// The bits of v under mask, as a float: q * 2^(shift - 149) for a nibble q at
// bit `shift` (shift <= 19), a subnormal number held exactly.
template <uint32_t MASK>
__device__ __forceinline__ float sub_nib(uint32_t v) {
    return __uint_as_float(v & MASK);
}

// The exact float -8 * 2^(s - 149): Q4_0's offset at nibble shift s.
__host__ __device__ constexpr uint32_t neg8_bits(int s) { return 0x80000000u | (8u << s); }

// Shift s (the power of two carried by the decoded value) of nibble position
// p = 0..7 of a word: positions 5..7 come from the word shifted right by 12.
__host__ __device__ constexpr int pos_shift(int p) { return p <= 4 ? 4 * p : 4 * (p - 3); }

// 2^e as a float for e in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float pow2f(int e) {
    return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(1u << (e + 149));
}

// ------------------------------------------------------------------ decode
// One word of eight nibbles as four packed pairs, Q4 order: a0 = (p0, p2),
// a1 = (p4, p6) are the low nibbles of bytes 0..3, b0 = (p1, p3),
// b1 = (p5, p7) the high nibbles. With kBias8 the exact offset 8 is removed.
// Loop-invariant packed constants, built once per thread (so that they stay
// in registers instead of being rematerialized at every use).
struct PairK {
    float2 bias[4];  // Q4_0: -8 * 2^(s-149) for the four decode pairs
    float2 inv[4];   // 2^-s of the four chains
};

template <bool kBias8>
__device__ __forceinline__ void dec_q4(uint32_t v, float2& a0, float2& a1, float2& b0, float2& b1,
                                       const PairK& k) {
    const uint32_t v2 = v >> 12;
    a0 = make_float2(sub_nib<0x0000Fu>(v), sub_nib<0x00F00u>(v));    // shifts 0, 8
    a1 = make_float2(sub_nib<0xF0000u>(v), sub_nib<0x0F000u>(v2));   // 16, 12
    b0 = make_float2(sub_nib<0x000F0u>(v), sub_nib<0x0F000u>(v));    // 4, 12
    b1 = make_float2(sub_nib<0x00F00u>(v2), sub_nib<0xF0000u>(v2));  // 8, 16
    if (kBias8) {
        a0 = __fadd2_rn(a0, k.bias[0]);
        a1 = __fadd2_rn(a1, k.bias[1]);
        b0 = __fadd2_rn(b0, k.bias[2]);
        b1 = __fadd2_rn(b1, k.bias[3]);
    }
}

// Packed affine word (code k = 8w + p at nibble p): pairs (p0,p1) (p2,p3)
// (p4,p5) (p6,p7), i.e. natural element order.
__device__ __forceinline__ void dec_packed(uint32_t v, float2& f0, float2& f1, float2& f2, float2& f3) {
    const uint32_t v2 = v >> 12;
    f0 = make_float2(sub_nib<0x0000Fu>(v), sub_nib<0x000F0u>(v));    // 0, 4
    f1 = make_float2(sub_nib<0x00F00u>(v), sub_nib<0x0F000u>(v));    // 8, 12
    f2 = make_float2(sub_nib<0xF0000u>(v), sub_nib<0x00F00u>(v2));   // 16, 8
    f3 = make_float2(sub_nib<0x0F000u>(v2), sub_nib<0xF0000u>(v2));  // 12, 16
}

// Two words of byte codes (k = 4w + t): each byte moved to bits 0..7 (the
// subnormal q * 2^-149), pairs in natural element order.
__device__ __forceinline__ void dec_u8(uint32_t va, uint32_t vb, float2& f0, float2& f1, float2& f2,
                                       float2& f3) {
    f0 = make_float2(__uint_as_float(__byte_perm(va, 0u, 0x4440)), __uint_as_float(__byte_perm(va, 0u, 0x4441)));
    f1 = make_float2(__uint_as_float(__byte_perm(va, 0u, 0x4442)), __uint_as_float(__byte_perm(va, 0u, 0x4443)));
    f2 = make_float2(__uint_as_float(__byte_perm(vb, 0u, 0x4440)), __uint_as_float(__byte_perm(vb, 0u, 0x4441)));
    f3 = make_float2(__uint_as_float(__byte_perm(vb, 0u, 0x4442)), __uint_as_float(__byte_perm(vb, 0u, 0x4443)));
}

// sa += (f0, f1) . xa and sb += (f2, f3) . xb: two independent chains of
// packed FMAs, in a fixed order.
__device__ __forceinline__ void dot8x2(float2& sa, float2& sb, const float2& f0, const float2& f1,
                                       const float2& f2, const float2& f3, const float4& xa,
                                       const float4& xb) {
    sa = __ffma2_rn(f0, make_float2(xa.x, xa.y), sa);
    sb = __ffma2_rn(f2, make_float2(xb.x, xb.y), sb);
    sa = __ffma2_rn(f1, make_float2(xa.z, xa.w), sa);
    sb = __ffma2_rn(f3, make_float2(xb.z, xb.w), sb);
}

// ------------------------------------------------------------ step compute
// Packed pair of the exact powers of two 2^-sa, 2^-sb (z is a runtime zero).
__device__ __forceinline__ float2 inv2(int sa, int sb, uint32_t z) {
    return make_float2(__uint_as_float(((uint32_t)(127 - sa) << 23) | z),
                       __uint_as_float(((uint32_t)(127 - sb) << 23) | z));
}

// The constants of format FMT; z is a runtime zero that keeps them from being
// folded back into every use.
template <int FMT>
__device__ __forceinline__ PairK make_pairk(uint32_t z) {
    PairK k;
    auto nb = [&](int sa, int sb) {
        return make_float2(__uint_as_float(neg8_bits(sa) | z), __uint_as_float(neg8_bits(sb) | z));
    };
    k.bias[0] = nb(0, 8);
    k.bias[1] = nb(16, 12);
    k.bias[2] = nb(4, 12);
    k.bias[3] = nb(8, 16);
    if (FMT == FMT_AFF_PACKED) {
        k.inv[0] = inv2(0, 4, z);
        k.inv[1] = inv2(8, 12, z);
        k.inv[2] = inv2(16, 8, z);
        k.inv[3] = inv2(12, 16, z);
    } else {
        k.inv[0] = inv2(0, 8, z);
        k.inv[1] = inv2(16, 12, z);
        k.inv[2] = inv2(4, 12, z);
        k.inv[3] = inv2(8, 16, z);
    }
    return k;
}

// One lane's unit of one step. xr[m] points at the lane's unit of staged x
// row m (natural order, element e in float4 e / 4, scaled by 2^c_m); xsr[m]
// at the unit's per-32 raw sums (two float4). Products are accumulated in
// float2 chains whose components each carry one fixed decode shift s; at the
// end of 32 weights the chains are multiplied by 2^-s (exact) and added.
// acc_s[m] collects the scaled products, acc_n[m] the offset terms (Q4_K
// min, affine bias) in natural units.
template <int FMT, int MT, int LPR>
__device__ __forceinline__ void step_unit(const uint8_t* __restrict__ slot, int lane, int sbl,
                                          int log2gs, const float4* const (&xr)[MT],
                                          const float4* const (&xsr)[MT], float (&acc_s)[MT],
                                          float (&acc_n)[MT], const PairK& k) {
    const float2 z2 = make_float2(0.0f, 0.0f);
    if constexpr (FMT == FMT_Q4_0) {
        const uint4* wp = reinterpret_cast<const uint4*>(slot + lane * 144);
        uint32_t W[36];
#pragma unroll
        for (int i = 0; i < 9; ++i) {
            const uint4 v = wp[i];
            W[4 * i] = v.x;
            W[4 * i + 1] = v.y;
            W[4 * i + 2] = v.z;
            W[4 * i + 3] = v.w;
        }
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            // The block's 16 nibble bytes as 4 words of bytes 4w..4w+3.
            uint32_t v[4], db;
            if ((b & 1) == 0) {  // block at byte 18b = 4 * (9b/2): d | q0 q1 | ... | q14 q15 d'
                const int base = 9 * b / 2;
#pragma unroll
                for (int wd = 0; wd < 4; ++wd) v[wd] = __byte_perm(W[base + wd], W[base + wd + 1], 0x5432);
                db = W[base] & 0xFFFFu;
            } else {             // block at byte 4 * (9b-1)/2 + 2: nibbles in 4 aligned words
                const int base = (9 * b + 1) / 2;
#pragma unroll
                for (int wd = 0; wd < 4; ++wd) v[wd] = W[base + wd];
                db = W[base - 1] >> 16;
            }
            const float d = __half2float(__ushort_as_half((unsigned short)db));
            float2 A0[MT], A1[MT], B0[MT], B1[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) A0[m] = A1[m] = B0[m] = B1[m] = z2;
#pragma unroll
            for (int wd = 0; wd < 4; ++wd) {
                float2 a0, a1, b0, b1;
                dec_q4<true>(v[wd], a0, a1, b0, b1, k);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float4 xa = xr[m][8 * b + wd], xb = xr[m][8 * b + 4 + wd];
                    A0[m] = __ffma2_rn(a0, make_float2(xa.x, xa.y), A0[m]);
                    A1[m] = __ffma2_rn(a1, make_float2(xa.z, xa.w), A1[m]);
                    B0[m] = __ffma2_rn(b0, make_float2(xb.x, xb.y), B0[m]);
                    B1[m] = __ffma2_rn(b1, make_float2(xb.z, xb.w), B1[m]);
                }
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float2 T = __fmul2_rn(A0[m], k.inv[0]);
                T = __ffma2_rn(A1[m], k.inv[1], T);
                T = __ffma2_rn(B0[m], k.inv[2], T);
                T = __ffma2_rn(B1[m], k.inv[3], T);
                acc_s[m] = __fmaf_rn(d, T.x + T.y, acc_s[m]);
            }
        }
    } else if constexpr (FMT == FMT_Q4_K) {
        const uint8_t* up = slot + lane * 144;
        const uint4 H = *reinterpret_cast<const uint4*>(up);
        const float d = __half2float(__ushort_as_half((unsigned short)(H.x & 0xFFFFu)));
        const float dm = __half2float(__ushort_as_half((unsigned short)(H.x >> 16)));
        // 6-bit (scale, min) of sub-blocks 0..3 and 4..7, one per byte.
        const uint32_t sc_lo = H.y & 0x3F3F3F3Fu, mn_lo = H.z & 0x3F3F3F3Fu;
        const uint32_t sc_hi = (H.w & 0x0F0F0F0Fu) | ((H.y >> 2) & 0x30303030u);
        const uint32_t mn_hi = ((H.w >> 4) & 0x0F0F0F0Fu) | ((H.z >> 2) & 0x30303030u);
        float4 sx0[MT], sx1[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            sx0[m] = xsr[m][0];
            sx1[m] = xsr[m][1];
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const uint32_t scw = cc < 2 ? sc_lo : sc_hi, mnw = cc < 2 ? mn_lo : mn_hi;
            const int sh = 16 * (cc & 1);
            const float a0 = d * (float)((scw >> sh) & 0xFFu);
            const float a1 = d * (float)((scw >> (sh + 8)) & 0xFFu);
            const float m0 = dm * (float)((mnw >> sh) & 0xFFu);
            const float m1 = dm * (float)((mnw >> (sh + 8)) & 0xFFu);
            const uint4 q0 = *reinterpret_cast<const uint4*>(up + 16 + 32 * cc);
            const uint4 q1 = *reinterpret_cast<const uint4*>(up + 32 + 32 * cc);
            const uint32_t v[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
            float2 A0[MT], A1[MT], B0[MT], B1[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) A0[m] = A1[m] = B0[m] = B1[m] = z2;
#pragma unroll
            for (int wd = 0; wd < 8; ++wd) {
                float2 pa0, pa1, pb0, pb1;
                dec_q4<false>(v[wd], pa0, pa1, pb0, pb1, k);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float4 xa = xr[m][16 * cc + wd], xb = xr[m][16 * cc + 8 + wd];
                    A0[m] = __ffma2_rn(pa0, make_float2(xa.x, xa.y), A0[m]);
                    A1[m] = __ffma2_rn(pa1, make_float2(xa.z, xa.w), A1[m]);
                    B0[m] = __ffma2_rn(pb0, make_float2(xb.x, xb.y), B0[m]);
                    B1[m] = __ffma2_rn(pb1, make_float2(xb.z, xb.w), B1[m]);
                }
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float2 L = __fmul2_rn(A0[m], k.inv[0]);
                L = __ffma2_rn(A1[m], k.inv[1], L);
                float2 Hh = __fmul2_rn(B0[m], k.inv[2]);
                Hh = __ffma2_rn(B1[m], k.inv[3], Hh);
                const float4 sx = cc < 2 ? sx0[m] : sx1[m];
                const float s_lo = (cc & 1) ? sx.z : sx.x, s_hi = (cc & 1) ? sx.w : sx.y;
                acc_s[m] = __fmaf_rn(a1, Hh.x + Hh.y, __fmaf_rn(a0, L.x + L.y, acc_s[m]));
                acc_n[m] = __fmaf_rn(-m1, s_hi, __fmaf_rn(-m0, s_lo, acc_n[m]));
            }
        }
    } else {
        constexpr int UB = Fmt<FMT>::UB;
        const uint8_t* up = slot + lane * UB;
        const float* sp = reinterpret_cast<const float*>(slot + 32 * UB + lane * sbl);
        const float* bp = reinterpret_cast<const float*>(slot + 32 * UB + 32 * sbl + lane * sbl);
        float4 sx0[MT], sx1[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            sx0[m] = xsr[m][0];
            sx1[m] = xsr[m][1];
        }
#pragma unroll
        for (int sg = 0; sg < 8; ++sg) {  // 32-code segments
            uint32_t v[8];
            if constexpr (FMT == FMT_AFF_PACKED) {
                const uint4 q = *reinterpret_cast<const uint4*>(up + 16 * sg);
                v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
            } else {
                const uint4 q0 = *reinterpret_cast<const uint4*>(up + 32 * sg);
                const uint4 q1 = *reinterpret_cast<const uint4*>(up + 32 * sg + 16);
                v[0] = q0.x; v[1] = q0.y; v[2] = q0.z; v[3] = q0.w;
                v[4] = q1.x; v[5] = q1.y; v[6] = q1.z; v[7] = q1.w;
            }
            float2 C0[MT], C1[MT], C2[MT], C3[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) C0[m] = C1[m] = C2[m] = C3[m] = z2;
#pragma unroll
            for (int wd = 0; wd < 4; ++wd) {
                float2 f0, f1, f2, f3;
                if constexpr (FMT == FMT_AFF_PACKED)
                    dec_packed(v[wd], f0, f1, f2, f3);
                else
                    dec_u8(v[2 * wd], v[2 * wd + 1], f0, f1, f2, f3);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float4 xa = xr[m][8 * sg + 2 * wd], xb = xr[m][8 * sg + 2 * wd + 1];
                    C0[m] = __ffma2_rn(f0, make_float2(xa.x, xa.y), C0[m]);
                    C1[m] = __ffma2_rn(f1, make_float2(xa.z, xa.w), C1[m]);
                    C2[m] = __ffma2_rn(f2, make_float2(xb.x, xb.y), C2[m]);
                    C3[m] = __ffma2_rn(f3, make_float2(xb.z, xb.w), C3[m]);
                }
            }
            const int gi = (sg << 5) >> log2gs;  // the segment's group within the unit
            const float sv = sp[gi], bv = bp[gi];
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                // Packed chains carry shifts (0,4) (8,12) (16,8) (12,16); byte codes
                // none. Scaling a chain by its exact 2^-s first makes both storages
                // add the same values in the same order.
                float2 T;
                if constexpr (FMT == FMT_AFF_PACKED) {
                    T = __fmul2_rn(C0[m], k.inv[0]);
                    T = __ffma2_rn(C1[m], k.inv[1], T);
                    T = __ffma2_rn(C2[m], k.inv[2], T);
                    T = __ffma2_rn(C3[m], k.inv[3], T);
                } else {
                    T = C0[m];
                    T = __fadd2_rn(C1[m], T);
                    T = __fadd2_rn(C2[m], T);
                    T = __fadd2_rn(C3[m], T);
                }
                const float4 sx = sg < 4 ? sx0[m] : sx1[m];
                const int k4 = sg & 3;
                const float xsg = k4 == 0 ? sx.x : k4 == 1 ? sx.y : k4 == 2 ? sx.z : sx.w;
                acc_s[m] = __fmaf_rn(sv, T.x + T.y, acc_s[m]);
                acc_n[m] = __fmaf_rn(bv, xsg, acc_n[m]);
            }
        }
    }
}

// ------------------------------------------------------------------ kernel
__device__ __forceinline__ int wi_c(int task, int tasks_per_w) { return task >= tasks_per_w ? 1 : 0; }

// Shared memory: x staged [MT][K/256 units][65 float4] (natural order,
// scaled by 2^c_m), raw x sums [MT][K/256][12] (8 used; formats with an
// offset term), per-warp max|x| of each input row ([2][16] words), then the
// warps' rings of S slots.
template <int FMT, int MT, int LPR>
__global__ void __launch_bounds__(256, 2) gemv_stream_kernel(const Params p) {
    using F = Fmt<FMT>;
    constexpr int UB = F::UB;
    constexpr int RW = 32 / LPR;           // rows per step
    constexpr int PIECES = UB / 16;        // 16-byte copies per lane per step
    constexpr int SEG_PIECES = LPR * UB / 16;  // pieces per row segment of a step
    constexpr bool kAffine = (FMT == FMT_AFF_U8 || FMT == FMT_AFF_PACKED);

    extern __shared__ __align__(128) uint8_t smem[];
    float* xs = reinterpret_cast<float*>(smem);
    float* xsum = reinterpret_cast<float*>(smem + p.xs_bytes);
    unsigned* wmax = reinterpret_cast<unsigned*>(smem + p.xs_bytes + p.xsum_bytes);
    uint8_t* ring = smem + p.xs_bytes + p.xsum_bytes + 128;

    const int nwarps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // CTA b takes tasks_base tasks, plus one more when b < tasks_rem.
    const int c_begin = (int)blockIdx.x * p.tasks_base + min((int)blockIdx.x, p.tasks_rem);
    const int c_end = c_begin + p.tasks_base + ((int)blockIdx.x < p.tasks_rem ? 1 : 0);

    // L2 prefetch of this CTA's rows (codes, and the affine scales/biases).
    auto prefetch_share = [&]() {
        for (int wi = 0; wi < p.nw; ++wi) {
            const int lo = max(c_begin, wi * p.tasks_per_w);
            const int hi = min(c_end, (wi + 1) * p.tasks_per_w);
            if (lo >= hi) continue;
            const long long r0 = (long long)(lo - wi * p.tasks_per_w) * RW;
            const long long r1 = min((long long)(hi - wi * p.tasks_per_w) * RW, (long long)p.N);
            const uint8_t* base = (wi == 0 ? p.w[0] : p.w[1]) + r0 * p.row_bytes;
            long long bytes = (r1 - r0) * p.row_bytes;
            for (long long off = 0; off < bytes; off += (1ll << 20))
                prefetch_l2(base + off, (uint32_t)min(bytes - off, 1ll << 20));
            if (kAffine) {
                const float* arr[2] = {p.s, p.b};
#pragma unroll
                for (int a = 0; a < 2; ++a) {
                    const uintptr_t s0 = reinterpret_cast<uintptr_t>(arr[a] + r0 * p.G);
                    const uintptr_t s1 = reinterpret_cast<uintptr_t>(arr[a] + r1 * p.G);
                    const uintptr_t a0 = (s0 + 15) & ~(uintptr_t)15, a1 = s1 & ~(uintptr_t)15;
                    if (a1 > a0) prefetch_l2(reinterpret_cast<const void*>(a0), (uint32_t)(a1 - a0));
                }
            }
        }
    };
    if (threadIdx.x == 0) prefetch_share();

    // This warp's tasks: c_begin + warp + i * nwarps.
    const int first = c_begin + warp;
    int ntask = 0;  // tasks first, first + nwarps, ... below c_end
    for (int tk = first; tk < c_end; tk += nwarps) ++ntask;
    const int nsteps = ntask * p.tpr;
    uint8_t* myring = ring + (size_t)warp * p.S * p.slot_bytes;
    const int ul = lane % LPR;

    // The lane's copy pieces of a step (the same for every step): piece k is
    // bytes [16q, 16q + 16) of the slot, q = lane + 32k, which come from row
    // segment q / SEG_PIECES of the step.
    int src_off[PIECES];
#pragma unroll
    for (int k = 0; k < PIECES; ++k) {
        const int q = lane + 32 * k;
        const int seg = q / SEG_PIECES;
        src_off[k] = seg * (int)p.row_bytes + (q - seg * SEG_PIECES) * 16;
    }
    // Affine: the lane's scale/bias bytes per unit and their offset in a row.
    const int sb_bytes = kAffine ? (p.log2gs >= 8 ? 4 : (1024 >> p.log2gs)) : 0;

    // Issue state: task i_task = (wi_i, rg_i), step t_i.
    int i_task = 0, t_i = 0;
    int wi_i = wi_c(first, p.tasks_per_w), rg_i = first - wi_i * p.tasks_per_w;
    // Copy the next step into slot `sl`; always commits one group (empty past
    // the end) so that group counting stays uniform.
    auto issue_next = [&](int sl) {
        if (i_task < ntask) {
            const int row0 = rg_i * RW;
            const uint8_t* base = (wi_i == 0 ? p.w[0] : p.w[1]) + (long long)row0 * p.row_bytes +
                                  (long long)t_i * (LPR * UB);
            const uint32_t dst = smem_addr(myring + (size_t)sl * p.slot_bytes) + 16 * lane;
            const int rows_left = p.N - row0;
            if (rows_left >= RW && p.tpr == 1) {
                // Whole rows: the step is one contiguous range.
                const uint8_t* src = base + 16 * lane;
#pragma unroll
                for (int k = 0; k < PIECES; ++k) cp_async16(dst + 512 * k, src + 512 * k);
            } else if (rows_left >= RW) {
#pragma unroll
                for (int k = 0; k < PIECES; ++k) cp_async16(dst + 512 * k, base + src_off[k]);
            } else {
#pragma unroll
                for (int k = 0; k < PIECES; ++k)
                    if ((lane + 32 * k) / SEG_PIECES < rows_left)
                        cp_async16(dst + 512 * k, base + src_off[k]);
            }
            if (kAffine) {
                const int r = row0 + lane / LPR;
                const int u = t_i * LPR + ul;
                if (r < p.N) {
                    const long long go = (long long)r * p.G + ((u * 256) >> p.log2gs);
                    const uint32_t d0 = smem_addr(myring + (size_t)sl * p.slot_bytes + 32 * UB + lane * p.sbl);
                    const uint32_t d1 = d0 + 32 * p.sbl;
                    if (sb_bytes >= 16) {
                        cp_async16(d0, p.s + go);
                        cp_async16(d1, p.b + go);
                        if (sb_bytes == 32) {
                            cp_async16(d0 + 16, p.s + go + 4);
                            cp_async16(d1 + 16, p.b + go + 4);
                        }
                    } else if (sb_bytes == 8) {
                        cp_async8(d0, p.s + go);
                        cp_async8(d1, p.b + go);
                    } else {
                        cp_async4(d0, p.s + go);
                        cp_async4(d1, p.b + go);
                    }
                }
            }
            if (++t_i == p.tpr) {
                t_i = 0;
                ++i_task;
                rg_i += nwarps;
                while (rg_i >= p.tasks_per_w) {
                    rg_i -= p.tasks_per_w;
                    ++wi_i;
                }
            }
        }
        cp_commit();
    };

    // The weights stream into L2 (prefetch above) while this kernel waits for
    // the preceding one; x may be produced by that kernel. The ring is filled
    // only after x is staged, so that x's loads do not queue behind it.
    pdl_launch_dependents();
    pdl_wait();

    // ---------------------------------------------------------- stage x
    // Pass 0: x, coalesced, into shared memory in natural order, unit by unit
    // with one float4 of padding per unit (reading a float4 of 8 consecutive
    // units is then bank-conflict free); the raw sum of every 32-element
    // segment (((x0 + x1) + x2) + x3 per float4, then an xor tree over the
    // segment's 8 lanes); max|x| per input row (as bits).
    // Pass 1: every staged float4 multiplied by 2^c_m (from registers when x
    // fits one round of loads, else in place).
    const int K4 = p.K >> 2;
    const int U = p.K >> 8;
    const int total4 = MT * K4;
    const float4* x4 = reinterpret_cast<const float4*>(p.x);
    float4* xw = reinterpret_cast<float4*>(xs);
    unsigned mx[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) mx[m] = 0;
    // One round of at most 8 float4 per thread keeps x in registers across the
    // max reduction; larger x goes through shared memory twice.
    const bool in_regs = total4 <= 8 * (int)blockDim.x;
    float4 v[8];
    for (int q0 = 0; q0 < total4; q0 += 8 * (int)blockDim.x) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int q = q0 + k * (int)blockDim.x + (int)threadIdx.x;
            v[k] = q < total4 ? __ldcg(x4 + q) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (q0 + k * (int)blockDim.x >= total4) break;  // uniform over the block
            const int q = q0 + k * (int)blockDim.x + (int)threadIdx.x;
            const bool ok = q < total4;
            const int mu = q >> 6;  // m * U + unit
            if (ok && !in_regs) xw[mu * 65 + (q & 63)] = v[k];
            const uint32_t a = max(max(__float_as_uint(v[k].x) & 0x7FFFFFFFu, __float_as_uint(v[k].y) & 0x7FFFFFFFu),
                                   max(__float_as_uint(v[k].z) & 0x7FFFFFFFu, __float_as_uint(v[k].w) & 0x7FFFFFFFu));
            const int m = (MT == 1 || q < K4) ? 0 : 1;
#pragma unroll
            for (int mm = 0; mm < MT; ++mm)
                if (mm == m) mx[mm] = max(mx[mm], a);
            if (F::kSums) {
                float sm = ((v[k].x + v[k].y) + v[k].z) + v[k].w;
                sm += __shfl_xor_sync(0xffffffffu, sm, 1);
                sm += __shfl_xor_sync(0xffffffffu, sm, 2);
                sm += __shfl_xor_sync(0xffffffffu, sm, 4);
                if (ok && (q & 7) == 0) xsum[mu * 12 + ((q & 63) >> 3)] = sm;
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        mx[m] = __reduce_max_sync(0xffffffffu, mx[m]);
        if (lane == 0) wmax[m * 16 + warp] = mx[m];
    }
    __syncthreads();

    // Per input row m: c_m = 119 - floor(log2 max|x_m|), clamped to [0, 127].
    int cexp[MT];
    float xmul[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        unsigned mall = 0;
        for (int w = 0; w < nwarps; ++w) mall = max(mall, wmax[m * 16 + w]);
        cexp[m] = min(127, max(0, 119 - ((int)(mall >> 23) - 127)));
        xmul[m] = __uint_as_float((uint32_t)(cexp[m] + 127) << 23);
    }
    auto scaled = [&](float4 u, int q) {
        const float f = (MT == 1 || q < K4) ? xmul[0] : xmul[MT - 1];
        return make_float4(__fmul_rn(u.x, f), __fmul_rn(u.y, f), __fmul_rn(u.z, f), __fmul_rn(u.w, f));
    };
    if (in_regs) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k * (int)blockDim.x >= total4) break;
            const int q = k * (int)blockDim.x + (int)threadIdx.x;
            if (q < total4) xw[(q >> 6) * 65 + (q & 63)] = scaled(v[k], q);
        }
    } else {
        for (int q = threadIdx.x; q < total4; q += blockDim.x) {
            float4& r = xw[(q >> 6) * 65 + (q & 63)];
            r = scaled(r, q);
        }
    }
    __syncthreads();

    // ------------------------------------------------------------ stream
    for (int q = 0; q < p.S; ++q) issue_next(q);
    float un1[MT], un2[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const int E = 149 - cexp[m];
        un1[m] = pow2f(min(E, 127));
        un2[m] = pow2f(E - min(E, 127));
    }
    const float4* xs4 = reinterpret_cast<const float4*>(xs);
    const float4* xsum4 = reinterpret_cast<const float4*>(xsum);
    const PairK pk = make_pairk<FMT>(p.zero);
    float acc_s[MT], acc_n[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc_s[m] = acc_n[m] = 0.0f;
    int t = 0, sl = 0;
    int wi = wi_c(first, p.tasks_per_w), rg = first - wi * p.tasks_per_w;
    for (int g = 0; g < nsteps; ++g) {
        cp_wait(p.S - 1);
        __syncwarp();
        const float4* xr[MT];
        const float4* xsr[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const int mu = m * U + t * LPR + ul;
            xr[m] = xs4 + mu * 65;
            xsr[m] = xsum4 + mu * 3;
        }
        step_unit<FMT, MT, LPR>(myring + (size_t)sl * p.slot_bytes, lane, p.sbl, p.log2gs, xr, xsr,
                                acc_s, acc_n, pk);
        __syncwarp();
        issue_next(sl);
        if (++sl == p.S) sl = 0;
        if (++t == p.tpr) {
            const int r = rg * RW + lane / LPR;
            float* out = wi == 0 ? p.out[0] : p.out[1];
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                // The lane's sum in natural units (exact power-of-two unscaling), then
                // the row's LPR lanes added with an xor butterfly.
                float v = __fadd_rn(__fmul_rn(__fmul_rn(acc_s[m], un1[m]), un2[m]), acc_n[m]);
#pragma unroll
                for (int off = LPR / 2; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (ul == 0 && r < p.N && m < p.M) out[(long long)m * p.N + r] = v;
                acc_s[m] = acc_n[m] = 0.0f;
            }
            t = 0;
            rg += nwarps;
            while (rg >= p.tasks_per_w) {
                rg -= p.tasks_per_w;
                ++wi;
            }
        }
    }
}

// Launch with programmatic stream serialization when pdl is set.
template <int FMT, int MT, int LPR>
int launch(const DevCtx& dc, const Params& kp, int grid, int warps, int smem, bool pdl,
           cudaStream_t s) {
    auto kern = gemv_stream_kernel<FMT, MT, LPR>;
    static int configured[64] = {0};
    cudaError_t e;
    if (dc.device < 0 || dc.device >= 64 || configured[dc.device] < smem) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dc.max_smem_optin);
        if (e != cudaSuccess) return cuda_fail(e);
        if (dc.device >= 0 && dc.device < 64) configured[dc.device] = dc.max_smem_optin;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(warps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, kp);
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

template <int FMT>
int dispatch(const DevCtx& dc, const Params& kp, int MT, int LPR, int grid, int warps, int smem, bool pdl, cudaStream_t s) {
#define QG_STREAM_LPR(MT_)                                                          \
    switch (LPR) {                                                                  \
        case 4: return launch<FMT, MT_, 4>(dc, kp, grid, warps, smem, pdl, s);          \
        case 8: return launch<FMT, MT_, 8>(dc, kp, grid, warps, smem, pdl, s);          \
        case 16: return launch<FMT, MT_, 16>(dc, kp, grid, warps, smem, pdl, s);        \
        default: return launch<FMT, MT_, 32>(dc, kp, grid, warps, smem, pdl, s);        \
    }
    if (MT == 1) {
        QG_STREAM_LPR(1)
    } else {
        QG_STREAM_LPR(2)
    }
#undef QG_STREAM_LPR
}

}  // namespace stream
}  // namespace qg
