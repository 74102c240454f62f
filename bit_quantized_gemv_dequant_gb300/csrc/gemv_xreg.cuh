// GEMV for one, two or four input rows with x held in registers, included by
// one translation unit per weight format.
//
// Pages: fused_dual_proj_q4_0.rs (mlx-native 0.9.1), q4_k_gemv_v2.rs
// (ferrum-kernels 0.7.7) and qmm_affine.rs (mlx-native 0.21.1) define the
// operations, the last one also the prepared AF4-g64 layout
// (prepare_af4_g64); the design below is for sm_103a.
//
//  * Lane <-> K unit. Every consumer lane owns one fixed unit of 32 weights
//    along K (a Q4_0 block; half of a Q4_K 32-byte nibble chunk, i.e. 16
//    elements of each of two sub-blocks; 32 affine codes; an AF4 32-group)
//    for the whole call.
//    Its 32 x values (per input row) are loaded once, pre-scaled, and stay in
//    registers; the lane then walks every weight row of its CTA's share. A
//    row group of WG warps covers one row's K; the NRG = NWC / WG row groups
//    of a CTA split the rows of each chunk.
//  * Q4_0 blocks are 18 bytes, so half of them start 2 bytes into a 32-bit
//    word. Warp w of a row group takes the blocks of one parity (w & 1), so
//    every lane of a warp runs the same code with compile-time word offsets,
//    and lanes read 36 bytes apart (conflict-free 32-bit shared loads).
//  * Exact decode, one instruction per nibble: a nibble masked in place in
//    its word, (word & 0xF << 4p), read as an f32 is the subnormal
//    q * 2^(4p - 149) exactly (p <= 4; the three upper nibbles use the word
//    shifted right by 12). Bytes (u8 codes) are moved to byte 0 by PRMT and
//    read as q * 2^-149. The matching x value was multiplied by
//    2^(S - 4p') when it was loaded, so every packed f32x2 FMA adds
//    q * x * 2^(S - 149) with a single rounding. S is one power of two per
//    input row for the whole grid, from max|x|, so that these products are
//    normal numbers: S = 126 - floor(log2 max|x|), clamped to [0, 127].
//  * Offsets and scales per unit: Q4_0's -8 is the chain's start value
//    -8 * sum(x) (scaled alike), then y += d * chain. Q4_K: the two lanes of a
//    chunk half-pair swap one chain each, so each lane ends with the 32-element
//    chain of one sub-block and applies (d * sc) and -(dmin * m) * sum(x) of
//    that sub-block (the scale pair it decodes itself, 6-bit fields by PRMT).
//    Affine and AF4: y += s * chain + b * sum(x) per group (AF4: bf16 scale
//    and bias of the unit's 64-group).
//  * Weights stream into a ring of shared-memory slots, one 1-D TMA bulk copy
//    per chunk of up to RC consecutive rows of one matrix (plus the chunk's
//    scales and biases for the affine format), issued by one producer lane
//    with an evict-first L2 policy and completing on mbarriers. AF4 chunks
//    (4 or 8 rows of one 64-row block across all of K) are two 2-D tensor
//    copies instead, the plane's with a 64- or 128-byte swizzle. CTAs take
//    contiguous, balanced ranges of rows (the dual projection's row list is
//    W_a then W_b), so the grid is balanced to one row (AF4: to four rows).
//  * Reduction: each lane has one value per (input row, chunk row of its
//    group); a transposing butterfly adds them across the warp, and the WG
//    warps of the group add their partial sums in warp order through shared
//    memory. The result is multiplied by 2^(149 - S) (exact) and stored.
//  * Programmatic dependent launch: the producer issues the first weight
//    copies before the kernel waits for its predecessor; consumers wait
//    (griddepcontrol.wait) before they read x and before any y is written.
//    With eight or twelve consumer warps and M = 1 the CTA uses at most half
//    an SM's registers and shared memory (four warps: a quarter), so the next
//    call's CTA can stream its weights while this one computes.
//
// Every output's arithmetic depends only on (format, M, K, x), never on N, the
// matrix count, the grid or the chunk: the dual projection is bitwise equal to
// two single projections.
#pragma once

#include <cuda_fp16.h>

#include "prefill_common.cuh"
#include "qg_internal.cuh"

namespace qg {
namespace xreg {

struct Params {
    const uint8_t* w[2];
    float* out[2];
    const float* x;
    const float* s;            // affine scales [N, G]
    const float* b;            // affine biases [N, G]
    int M, N, K, nw;
    int log2gs, G;
    int row_bytes;             // code bytes of one weight row
    int rows_base, rows_rem;   // CTA c takes rows_base units of rows, one more when c < rows_rem
    int row_unit;              // rows per unit (0 or 1: single rows; AF4: 4, so chunks start
                               // on 4-row boundaries as its metadata copies require)
    int S, slot_bytes;         // ring slots and their size
    int sb_off;                // offset of the chunk's scales in a slot (biases follow)
    int WG, NRG, RC;           // warps per row group, row groups, rows per chunk
    int units;                 // valid lane units per row (Q4_0: blocks)
    int rbuf;                  // rows of per-warp partial sums buffered before a flush
    int red_floats;            // floats of the partial-sum region (a multiple of 4)
    int ahead;                 // chunks in flight at most (0: the whole ring)
    int dep_wait;              // 1: wait for the preceding kernel before reading x / writing y
    unsigned* err;
};

// 2^n as an f32, for n in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float pow2f(int n) {
    return n >= -126 ? __uint_as_float((uint32_t)(n + 127) << 23)
                     : __uint_as_float(1u << (n + 149));
}

// Nibble at position pos (bits 4pos..4pos+3) of v as the exact subnormal
// q * 2^(nib_shift(pos) - 149).
// (The word shifted right by 12 comes from the high half of v * 2^20, an
// integer multiply that runs beside the logic unit that does the masking.)
__device__ __forceinline__ float nib(uint32_t v, int pos) {
    return pos <= 4 ? __uint_as_float(v & (0xFu << (4 * pos)))
                    : __uint_as_float(__umulhi(v, 1u << 20) & (0xFu << (4 * (pos - 3))));
}
__host__ __device__ constexpr int nib_shift(int pos) { return pos <= 4 ? 4 * pos : 4 * (pos - 3); }

// Where the two elements (2k, 2k+1) of pair k of a lane unit sit: word index
// and the two nibble positions (or byte positions, u8) in that word.
struct Loc {
    int word, pa, pb;
};

// Q4_0 block with parity par: the block starts 0 (even) or 2 (odd) bytes into
// its first word; qs byte i holds element i (low nibble) and 16 + i (high).
// Pairs 0..7 are the low nibbles of bytes 2k, 2k+1; pairs 8..15 the high ones.
__host__ __device__ constexpr Loc q40_loc(int par, int k) {
    return Loc{((par ? 4 : 2) + 2 * (k & 7)) >> 2,
               2 * (((par ? 4 : 2) + 2 * (k & 7)) & 3) + (k >= 8 ? 1 : 0),
               2 * (((par ? 4 : 2) + 2 * (k & 7)) & 3) + 2 + (k >= 8 ? 1 : 0)};
}
// Q4_K unit (16 nibble bytes): byte i holds element i of the low sub-block
// (low nibble) and of the high sub-block (high nibble). Pairs 0..7: low.
__host__ __device__ constexpr Loc q4k_loc(int k) {
    return Loc{(2 * (k & 7)) >> 2, 2 * ((2 * (k & 7)) & 3) + (k >= 8 ? 1 : 0),
               2 * ((2 * (k & 7)) & 3) + 2 + (k >= 8 ? 1 : 0)};
}
// Packed affine unit (16 bytes, 32 codes): element e = nibble e % 8 of word e / 8.
__host__ __device__ constexpr Loc packed_loc(int k) { return Loc{k >> 2, 2 * (k & 3), 2 * (k & 3) + 1}; }
// u8 affine unit (32 bytes): element e = byte e % 4 of word e / 4.
__host__ __device__ constexpr Loc u8_loc(int k) { return Loc{k >> 1, 2 * (k & 1), 2 * (k & 1) + 1}; }
// AF4-g64 unit (16 bytes, one 32-group of a row): word c holds, for p = 0..3,
// the element pair (16 (p >> 1) + 4c + 2 (p & 1), +1) in nibbles p and 4 + p.
// Pair k = elements (2k, 2k+1): c = (k & 7) >> 1, p = 2 (k >> 3) + (k & 1).
__host__ __device__ constexpr Loc af4_loc(int k) {
    return Loc{(k & 7) >> 1, 2 * (k >> 3) + (k & 1), 4 + 2 * (k >> 3) + (k & 1)};
}

// log2 of the power of two each decoded element of pair k carries (removed
// from x when x is loaded).
template <int FMT, int PAR>
__host__ __device__ constexpr int shift_a(int k) {
    return FMT == FMT_AFF_U8       ? 0
           : FMT == FMT_Q4_0       ? nib_shift(q40_loc(PAR, k).pa)
           : FMT == FMT_Q4_K       ? nib_shift(q4k_loc(k).pa)
           : FMT == FMT_AF4        ? nib_shift(af4_loc(k).pa)
                                   : nib_shift(packed_loc(k).pa);
}
template <int FMT, int PAR>
__host__ __device__ constexpr int shift_b(int k) {
    return FMT == FMT_AFF_U8       ? 0
           : FMT == FMT_Q4_0       ? nib_shift(q40_loc(PAR, k).pb)
           : FMT == FMT_Q4_K       ? nib_shift(q4k_loc(k).pb)
           : FMT == FMT_AF4        ? nib_shift(af4_loc(k).pb)
                                   : nib_shift(packed_loc(k).pb);
}

__device__ __forceinline__ float byte_f(uint32_t v, int t) {
    return __uint_as_float(__byte_perm(v, 0u, 0x4440u + (uint32_t)t));
}

// Decoded pair k of a unit whose words are wd.
template <int FMT, int PAR, int NWD>
__device__ __forceinline__ float2 pair(const uint32_t (&wd)[NWD], int k) {
    if (FMT == FMT_AFF_U8) {
        const Loc L = u8_loc(k);
        return make_float2(byte_f(wd[L.word], L.pa), byte_f(wd[L.word], L.pb));
    }
    const Loc L = FMT == FMT_Q4_0   ? q40_loc(PAR, k)
                  : FMT == FMT_Q4_K ? q4k_loc(k)
                  : FMT == FMT_AF4  ? af4_loc(k)
                                    : packed_loc(k);
    return make_float2(nib(wd[L.word], L.pa), nib(wd[L.word], L.pb));
}

// Warp reduction of V values at once; lane l ends with value l / (32 / V).
// Every value follows the same xor tree whatever V is.
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
                    // Both halves are added across the lane pair; the lower
                    // lane keeps the first, the upper lane the second (one
                    // select instead of two).
                    const float a = v[i] + __shfl_xor_sync(0xffffffffu, v[i], off);
                    const float b = v[i + half] + __shfl_xor_sync(0xffffffffu, v[i + half], off);
                    v[i] = upper ? b : a;
                }
            }
            cur = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
        }
    }
}

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// The chunk that starts at row r of the concatenated row list [rb, re).
struct Chunk {
    int wi, row0, n;
};
__device__ __forceinline__ Chunk chunk_at(int r, int re, int N, int RC) {
    const int wi = r >= N ? 1 : 0;
    const int row0 = r - wi * N;
    return Chunk{wi, row0, min(min(re - r, RC), N - row0)};
}
// AF4: a chunk also stays inside its 64-row block (one copy per block).
template <int FMT>
__device__ __forceinline__ Chunk chunk_of(int r, int re, int N, int RC) {
    if (FMT == FMT_AF4) return Chunk{0, r, min(min(re - r, RC), 64 - (r & 63))};
    return chunk_at(r, re, N, RC);
}

// The CTA's row range [rb, re).
__device__ __forceinline__ void cta_rows(const Params& p, int& rb, int& re) {
    const int cta = blockIdx.x, ru = max(1, p.row_unit);
    rb = ru * (cta * p.rows_base + min(cta, p.rows_rem));
    re = rb + ru * (p.rows_base + (cta < p.rows_rem ? 1 : 0));
}

// L2 prefetch of a 2-D tensor-map box (no completion to wait for).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

// All consumer threads load x with coalesced 16-byte loads into shared memory,
// laid out per lane unit (8 float4 chunks in the lane's pair order, chunk j
// stored at j ^ (reader lane & 7), so that the lanes' reads are
// conflict-free), and each warp writes its max |x| per input row to xmax.
template <int FMT, int MT, int NWC>
__device__ __forceinline__ void stage_x(const Params& p, float* xst, float* xmax, int warp,
                                        int lane) {
    const int nthr_all = NWC * 32, tid_all = warp * 32 + lane;
    float4* xs4 = reinterpret_cast<float4*>(xst);
    const int q4n = p.K >> 2;
    float amax[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        amax[m] = 0.0f;
        // A launch of four input rows may carry fewer (M = 3): the missing
        // rows are zeros, computed but never stored.
        const bool row_ok = m < p.M;
        const float4* xr = reinterpret_cast<const float4*>(p.x + (long long)(row_ok ? m : 0) * p.K);
        for (int q0 = tid_all; q0 < q4n; q0 += 4 * nthr_all) {
            float4 t[4];
#pragma unroll
            for (int i2 = 0; i2 < 4; ++i2) {
                const int q = q0 + i2 * nthr_all;
                t[i2] = (row_ok && q < q4n) ? xr[q] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i2 = 0; i2 < 4; ++i2) {
                const int q = q0 + i2 * nthr_all;
                if (q >= q4n) break;
                const int k = q << 2;
                int uq, jq;
                if (FMT == FMT_Q4_K) {
                    const int w = k & 255, r2 = w & 31;
                    uq = 8 * (k >> 8) + 2 * (w >> 6) + (r2 >> 4);
                    jq = 4 * ((w >> 5) & 1) + ((r2 & 15) >> 2);
                } else {
                    uq = k >> 5;
                    jq = (k & 31) >> 2;
                }
                const int key = (FMT == FMT_Q4_0 ? (uq >> 1) : uq) & 7;
                xs4[(size_t)m * (q4n) + uq * 8 + (jq ^ key)] = t[i2];
                amax[m] = fmaxf(amax[m], fmaxf(fmaxf(fabsf(t[i2].x), fabsf(t[i2].y)),
                                               fmaxf(fabsf(t[i2].z), fabsf(t[i2].w))));
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            amax[m] = fmaxf(amax[m], __shfl_xor_sync(0xffffffffu, amax[m], off));
        if (lane == 0) xmax[warp * MT + m] = amax[m];
    }
}

// Consumer warps of one Q4_0 parity class (PAR), or of another format (PAR 0).
template <int FMT, int MT, int NWC, int RPG, int PAR>
__device__ __forceinline__ void consume(const Params& p, uint8_t* ring, uint64_t* full,
                                       uint64_t* empty, float* red, float* xst, float* xmax,
                                       int warp, int lane) {
    constexpr int V = MT * RPG;
    constexpr bool kAffine = (FMT == FMT_AFF_U8 || FMT == FMT_AFF_PACKED);
    const int grp = warp / p.WG, gw = warp - grp * p.WG;
    const bool in_group = grp < p.NRG;

    // ------------------------------------------------- this lane's K unit
    int u;
    if (FMT == FMT_Q4_0) u = 64 * (gw >> 1) + 2 * lane + PAR;
    else u = gw * 32 + lane;
    // A lane past the end of a row (narrow K) gets x = 0 and reads a unit of
    // the row with its own layout (a Q4_0 block of its parity), so that it
    // adds exactly zero, or NaN only to a row whose exact result is not
    // finite anyway (a non-finite scale in that unit).
    const bool valid = in_group && u < p.units;
    const int uu = valid ? u : (FMT == FMT_Q4_0 ? PAR : 0);
    int qoff, hoff = 0;
    if (FMT == FMT_Q4_0) {
        qoff = (18 * uu) & ~3;
    } else if (FMT == FMT_Q4_K) {
        const int sb = uu >> 3, j = uu & 7;
        qoff = 144 * sb + 16 + 16 * j;
        hoff = 144 * sb;
    } else {
        qoff = (FMT == FMT_AFF_U8 ? 32 : 16) * uu;
    }
    const int grp_s = kAffine ? ((32 * uu) >> p.log2gs) : 0;
    // Q4_K: the scale pair this lane decodes (sub-block j = unit % 8) and the
    // constants that make the 6-bit field extraction branch-free.
    const int j8 = uu & 7, hh = uu & 1;
    const uint32_t k_mlo = j8 < 4 ? 63u : 15u, k_shm = j8 < 4 ? 0u : 4u;
    const uint32_t k_shh = j8 < 4 ? 0u : (uint32_t)(8 * j8 - 30), k_mh = j8 < 4 ? 0u : 0x30u;

    // x and y may be produced / consumed by the preceding kernel (unless the
    // caller declared the calls independent). x is staged while the producer
    // issues the weight copies.
    if (p.dep_wait) pdl_wait();
    stage_x<FMT, MT, NWC>(p, xst, xmax, warp, lane);
    const int q4n = p.K >> 2;
    const float4* xs4 = reinterpret_cast<const float4*>(xst);
    named_bar_sync(1, NWC * 32);
    int S_[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        float a = 0.0f;
        for (int w = 0; w < NWC; ++w) a = fmaxf(a, xmax[w * MT + m]);
        const int e = (int)((__float_as_uint(a) >> 23) & 0xFF);  // biased exponent
        S_[m] = max(0, min(127, 253 - e));
    }
    float xn[MT][32];
    {
        const int key = (FMT == FMT_Q4_0 ? (uu >> 1) : uu) & 7;
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 t = valid ? xs4[(size_t)m * q4n + uu * 8 + (j ^ key)]
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                xn[m][4 * j + 0] = t.x;
                xn[m][4 * j + 1] = t.y;
                xn[m][4 * j + 2] = t.z;
                xn[m][4 * j + 3] = t.w;
            }
    }
    if (!in_group) return;

    float2 X[MT][16];
    float xoff[MT];  // Q4_0: -8 sum(x); Q4_K, affine: sum(x) of the unit's group of elements
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const int S = S_[m];
#pragma unroll
        for (int k = 0; k < 16; ++k)
            X[m][k] = make_float2(xn[m][2 * k] * pow2f(S - shift_a<FMT, PAR>(k)),
                                  xn[m][2 * k + 1] * pow2f(S - shift_b<FMT, PAR>(k)));
        if (FMT == FMT_Q4_K) {
            float slo = 0.0f, shi = 0.0f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                slo += xn[m][j];
                shi += xn[m][16 + j];
            }
            const float plo = __shfl_xor_sync(0xffffffffu, slo, 1);
            const float phi = __shfl_xor_sync(0xffffffffu, shi, 1);
            const float sub = hh ? (shi + phi) : (slo + plo);
            xoff[m] = sub * pow2f(S - 149);
        } else {
            float sx = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) sx += xn[m][j];
            xoff[m] = FMT == FMT_Q4_0 ? -sx * pow2f(S - 146) : sx * pow2f(S - 149);
        }
    }
    // 2^(149 - S) in two factors (it exceeds the f32 range for S < 22).
    float dsc1[MT], dsc2[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const int t = 149 - S_[m];
        dsc1[m] = pow2f(min(t, 127));
        dsc2[m] = pow2f(t - min(t, 127));
    }

    // ------------------------------------------------------- chunk loop
    // Loop-invariant start values of the accumulator pairs.
    float2 acc0[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc0[m] = make_float2(FMT == FMT_Q4_0 ? xoff[m] : 0.0f, 0.0f);
    const float2 zero2 = make_float2(0.0f, 0.0f);
    int rb, re;
    cta_rows(p, rb, re);
    const int nthr = p.NRG * p.WG * 32, tid = warp * 32 + lane;
    // AF4: the 16-byte chunk of row rr of this lane's unit sits at rr ^ swz in
    // the unit's line of the slot (the copy's 64- or 128-byte swizzle).
    const int af4_swz = p.RC == 8 ? (uu & 7) : ((uu >> 1) & 3);
    const int NRG = p.NRG, RC = p.RC, WG = p.WG, N = p.N;
    const size_t row_bytes = (size_t)p.row_bytes;
    // Per-warp partial sums of the CTA's rows wait in red[row - fb][m][gw]
    // (rows fb .. fb + rbuf - 1) and are added in warp order when the buffer is
    // flushed: once at the end, or earlier whenever it would overflow.
    int fb = rb;
    // (After a wait gave up, the outputs are undefined: the error word tells.)
    auto flush = [&](int upto, bool last) {
        named_bar_sync(2, nthr);
        const int cnt = (upto - fb) * MT;
        for (int e = tid; e < cnt; e += nthr) {
            const int lr = e / MT, m = e - lr * MT;
            const float* src = red + (size_t)e * WG;
            float t = src[0];
            for (int g2 = 1; g2 < WG; ++g2) t += src[g2];
            const int ra = fb + lr;
            const int wi = ra >= N ? 1 : 0;
            if (m < p.M) p.out[wi][(long long)m * N + (ra - wi * N)] = t * dsc1[m] * dsc2[m];
        }
        if (!last) named_bar_sync(2, nthr);
        fb = upto;
    };
    bool dead = false;
    int slot = 0;
    uint32_t phase = 0;
    for (int r = rb; r < re;) {
        const Chunk ch = chunk_of<FMT>(r, re, N, RC);
        if (r + ch.n - fb > p.rbuf) flush(r, false);
        if (!dead && !mbar_wait(smem_addr(&full[slot]), phase)) {
            report_error(p.err, DEVERR_WAIT_FULL);
            dead = true;
        }
        const uint8_t* base = ring + (size_t)slot * p.slot_bytes;
        // Value(s) of row rr of the chunk for this lane's unit.
        auto row_value = [&](int rr, float (&o)[MT]) {
            const uint8_t* rowp = base + rr * row_bytes;
            if constexpr (FMT == FMT_Q4_0) {
                const uint32_t* wp = reinterpret_cast<const uint32_t*>(rowp + qoff);
                uint32_t wd[5];
#pragma unroll
                for (int t = 0; t < 5; ++t) wd[t] = wp[t];
                const __half2 dh = *reinterpret_cast<const __half2*>(&wd[0]);
                const float d = PAR ? __high2float(dh) : __low2float(dh);
                // Two chains (even and odd pairs) halve the dependent FMA depth.
                float2 acc[MT][2];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float2 f = pair<FMT, PAR, 5>(wd, k);
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        acc[m][k & 1] = __ffma2_rn(f, X[m][k], k == 0 ? acc0[m]
                                                              : k == 1 ? zero2 : acc[m][k & 1]);
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float2 t = __fadd2_rn(acc[m][0], acc[m][1]);
                    o[m] = d * (t.x + t.y);
                }
            } else if constexpr (FMT == FMT_Q4_K) {
                const uint4 qv = *reinterpret_cast<const uint4*>(rowp + qoff);
                const uint4 hd = *reinterpret_cast<const uint4*>(rowp + hoff);
                const uint32_t wd[4] = {qv.x, qv.y, qv.z, qv.w};
                float2 c0[MT], c1[MT];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float2 f = pair<FMT, 0, 4>(wd, k);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if (k < 8) c0[m] = __ffma2_rn(f, X[m][k], k == 0 ? acc0[m] : c0[m]);
                        else c1[m] = __ffma2_rn(f, X[m][k], k == 8 ? acc0[m] : c1[m]);
                    }
                }
                // (sc, m) of sub-block j8 as exact floats (2^23 + v, minus 2^23).
                const uint32_t MG = 0x4B000000u;
                const uint32_t scb = (__byte_perm(hd.y, hd.w, (uint32_t)j8) & k_mlo) |
                                     ((hd.y >> k_shh) & k_mh) | MG;
                const uint32_t mnb = ((__byte_perm(hd.z, hd.w, (uint32_t)j8) >> k_shm) & k_mlo) |
                                     ((hd.z >> k_shh) & k_mh) | MG;
                const float fsc = __uint_as_float(scb) - 8388608.0f;
                const float fmn = __uint_as_float(mnb) - 8388608.0f;
                const float d = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu)));
                const float dmin = __half2float(__ushort_as_half((unsigned short)(hd.x >> 16)));
                const float a = d * fsc, bm = dmin * fmn;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float s0 = c0[m].x + c0[m].y, s1 = c1[m].x + c1[m].y;
                    const float send = hh ? s0 : s1, mine = hh ? s1 : s0;
                    const float tot = mine + __shfl_xor_sync(0xffffffffu, send, 1);
                    o[m] = __fmaf_rn(a, tot, -(bm * xoff[m]));
                }
            } else if constexpr (FMT == FMT_AF4) {
                const uint4 q0 = *reinterpret_cast<const uint4*>(
                    base + ((size_t)uu * RC + (rr ^ af4_swz)) * 16);
                const uint32_t wd[4] = {q0.x, q0.y, q0.z, q0.w};
                // bf16 scale | bf16 bias << 16 of the unit's 64-group.
                const uint32_t mw = *reinterpret_cast<const uint32_t*>(
                    base + p.sb_off + ((size_t)(uu >> 1) * RC + rr) * 4);
                const float sc = __uint_as_float(mw << 16);
                const float bi = __uint_as_float(mw & 0xFFFF0000u);
                float2 acc[MT][2];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float2 f = pair<FMT, 0, 4>(wd, k);
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        acc[m][k & 1] = __ffma2_rn(f, X[m][k], k < 2 ? zero2 : acc[m][k & 1]);
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float2 t = __fadd2_rn(acc[m][0], acc[m][1]);
                    o[m] = __fmaf_rn(sc, t.x + t.y, bi * xoff[m]);
                }
            } else {
                constexpr int NWD = FMT == FMT_AFF_U8 ? 8 : 4;
                uint32_t wd[NWD];
                const uint4 q0 = *reinterpret_cast<const uint4*>(rowp + qoff);
                wd[0] = q0.x; wd[1] = q0.y; wd[2] = q0.z; wd[3] = q0.w;
                if constexpr (NWD == 8) {
                    const uint4 q1 = *reinterpret_cast<const uint4*>(rowp + qoff + 16);
                    wd[4] = q1.x; wd[5] = q1.y; wd[6] = q1.z; wd[7] = q1.w;
                }
                const float* sp = reinterpret_cast<const float*>(base + p.sb_off);
                const float sc = sp[rr * p.G + grp_s];
                const float bi = sp[(RC + rr) * p.G + grp_s];
                float2 acc[MT][2];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float2 f = pair<FMT, 0, NWD>(wd, k);
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        acc[m][k & 1] = __ffma2_rn(f, X[m][k], k < 2 ? zero2 : acc[m][k & 1]);
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float2 t = __fadd2_rn(acc[m][0], acc[m][1]);
                    o[m] = __fmaf_rn(sc, t.x + t.y, bi * xoff[m]);
                }
            }
        };
        // The group's RPG rows in one straight-line block, then one
        // transposing butterfly for all of them. In a short chunk (the end of
        // the CTA's range or of a matrix) the rows past its end are computed
        // from stale slot bytes and never stored.
        float v[V];
#pragma unroll
        for (int q = 0; q < RPG; ++q) {
            float o[MT];
            row_value(grp + q * NRG, o);
#pragma unroll
            for (int m = 0; m < MT; ++m) v[m * RPG + q] = o[m];
        }
        // The slot is free once every warp has read its rows.
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[slot]));
        butterfly<V>(v, lane);
        constexpr int kSpan = 32 / V;
        if ((lane % kSpan) == 0) {
            const int idx = lane / kSpan;
            const int m = idx / RPG, q = idx % RPG;
            const int rr = grp + q * NRG;
            if (rr < ch.n) red[((size_t)(r + rr - fb) * MT + m) * WG + gw] = v[0];
        }
        r += ch.n;
        if (++slot == p.S) {
            slot = 0;
            phase ^= 1u;
        }
    }
    flush(re, true);
}

// The kernel. mq / mm: AF4's tensor maps of the plane and the metadata
// (null for the other formats).
template <int FMT, int MT, int NWC, int RPG>
__device__ __forceinline__ void xreg_body(const Params& p, const CUtensorMap* mq,
                                          const CUtensorMap* mm) {
    extern __shared__ __align__(128) uint8_t smem[];
    // AF4's swizzled copies need their slots on 1024-byte boundaries (the
    // launch adds 1024 bytes for this).
    uint8_t* ring = FMT == FMT_AF4 ? smem + ((1024u - (smem_addr(smem) & 1023u)) & 1023u) : smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)p.S * p.slot_bytes);
    uint64_t* empty = full + p.S;
    float* red = reinterpret_cast<float*>(empty + p.S);
    float* xst = red + (size_t)p.red_floats;  // 16-byte aligned (red_floats % 4 == 0)
    float* xmax = xst + (size_t)MT * p.K;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int rb, re;
    cta_rows(p, rb, re);

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.S; ++i) {
            mbar_init(smem_addr(&full[i]), 1);
            mbar_init(smem_addr(&empty[i]), p.NRG * p.WG);
        }
        fence_mbar_init();
    }
    __syncthreads();

    // ------------------------------------------------------------ producer
    // Weights, scales and biases are read before griddepcontrol.wait: under
    // programmatic dependent launch they must not be written by the kernel
    // that precedes this one on the stream (the documented contract of that
    // launch mode). Without it the wait is a no-op.
    if (warp == NWC) {
        if (lane != 0) return;
        // The next kernel in the stream may be scheduled right away: it
        // waits for this one (griddepcontrol.wait) before touching anything
        // this one writes, and each bulk copy takes long to issue, so a
        // trigger after the first copies would delay the next launch by
        // microseconds.
        pdl_launch_dependents();
        const uint64_t pol = l2_evict_first();
        constexpr bool kAffine = (FMT == FMT_AFF_U8 || FMT == FMT_AFF_PACKED);
        int issued = 0;
        bool ok = true, prefetched = false;
        int i = 0;
        for (int r = rb; r < re; ++i) {
            const Chunk ch = chunk_of<FMT>(r, re, p.N, p.RC);
            r += ch.n;
            const int slot = i % p.S, use = i / p.S;
            if (use > 0 && !mbar_wait(smem_addr(&empty[slot]), (use - 1) & 1)) {
                report_error(p.err, DEVERR_WAIT_EMPTY);
                ok = false;
                break;
            }
            // At most `ahead` chunks in flight (ahead <= S, so the awaited
            // phase of chunk i - ahead is the latest one of its slot).
            if (p.ahead > 0 && i >= p.ahead) {
                const int j = i - p.ahead;
                if (!mbar_wait(smem_addr(&full[j % p.S]), (j / p.S) & 1)) {
                    report_error(p.err, DEVERR_WAIT_FULL);
                    ok = false;
                    break;
                }
            }
            uint8_t* dst = ring + (size_t)slot * p.slot_bytes;
            const uint32_t bar = smem_addr(&full[slot]);
            if constexpr (FMT == FMT_AF4) {
                // RC rows of the chunk's 64-row block, all 32-groups (codes)
                // and 64-groups (metadata): two tensor copies of fixed size
                // (rows past the block's end read as zeros, unused ones are
                // never stored).
                const uint32_t qb = (uint32_t)(p.RC * 16 * p.units);
                const uint32_t mb = (uint32_t)(p.RC * 4 * (p.units >> 1));
                mbar_arrive_expect_tx(bar, qb + mb);
                prefill::tma_load_2d(smem_addr(dst), mq, (ch.row0 & 63) * 16,
                                     (ch.row0 >> 6) * p.units, bar);
                prefill::tma_load_2d(smem_addr(dst + p.sb_off), mm, (ch.row0 & 63) * 4,
                                     (ch.row0 >> 6) * (p.units >> 1), bar);
            } else {
                const uint32_t qb = (uint32_t)(ch.n * p.row_bytes);
                const uint32_t sbb = kAffine ? (uint32_t)(ch.n * p.G * 4) : 0u;
                mbar_arrive_expect_tx(bar, qb + 2u * sbb);
                bulk_g2s(smem_addr(dst), p.w[ch.wi] + (long long)ch.row0 * p.row_bytes, qb, bar, pol);
                if (kAffine) {
                    const long long go = (long long)ch.row0 * p.G;
                    bulk_g2s(smem_addr(dst + p.sb_off), p.s + go, sbb, bar, pol);
                    bulk_g2s(smem_addr(dst + p.sb_off + p.RC * p.G * 4), p.b + go, sbb, bar, pol);
                }
            }
            issued = i + 1;
            if (i == p.S - 1 || r == re) {
                if (!prefetched && r < re && p.ahead == 0) {
                    // The rest of the CTA's rows does not fit in the ring:
                    // bring it from HBM into L2 now, so that the ring is later
                    // refilled at L2 latency.
                    for (int r2 = r; r2 < re;) {
                        const Chunk c2 = chunk_of<FMT>(r2, re, p.N, p.RC);
                        r2 += c2.n;
                        if constexpr (FMT == FMT_AF4) {
                            tma_prefetch_2d(mq, (c2.row0 & 63) * 16, (c2.row0 >> 6) * p.units);
                            tma_prefetch_2d(mm, (c2.row0 & 63) * 4, (c2.row0 >> 6) * (p.units >> 1));
                            continue;
                        }
                        bulk_prefetch_l2(p.w[c2.wi] + (long long)c2.row0 * p.row_bytes,
                                         (uint32_t)(c2.n * p.row_bytes));
                        if (kAffine) {
                            const long long go = (long long)c2.row0 * p.G;
                            bulk_prefetch_l2(p.s + go, (uint32_t)(c2.n * p.G * 4));
                            bulk_prefetch_l2(p.b + go, (uint32_t)(c2.n * p.G * 4));
                        }
                    }
                }
                prefetched = true;
            }
        }

        if (!ok) {
            // Let every slot's latest copy land before shared memory is released.
            for (int slot = 0; slot < p.S && slot < issued; ++slot) {
                const int last = slot + ((issued - 1 - slot) / p.S) * p.S;
                if (!mbar_wait(smem_addr(&full[slot]), (last / p.S) & 1))
                    report_error(p.err, DEVERR_WAIT_DRAIN);
            }
        }
        return;
    }

    // ----------------------------------------------------------- consumers
    if (FMT == FMT_Q4_0) {
        // Warp-uniform parity of the warp's blocks (warp index within its row group).
        if (((warp % p.WG) & 1) == 0)
            consume<FMT, MT, NWC, RPG, 0>(p, ring, full, empty, red, xst, xmax, warp, lane);
        else
            consume<FMT, MT, NWC, RPG, 1>(p, ring, full, empty, red, xst, xmax, warp, lane);
    } else {
        consume<FMT, MT, NWC, RPG, 0>(p, ring, full, empty, red, xst, xmax, warp, lane);
    }
}

#define QG_XREG_BOUNDS                                                      \
    __launch_bounds__((NWC + 1) * 32, MT == 4    ? 1                        \
                                      : NWC == 4 ? (MT == 1 ? 4 : 3)        \
                                      : ((NWC == 8 || NWC == 12) && MT == 1) ? 2 \
                                                                             : 1)

template <int FMT, int MT, int NWC, int RPG>
__global__ void QG_XREG_BOUNDS gemv_xreg_kernel(const Params p) {
    xreg_body<FMT, MT, NWC, RPG>(p, nullptr, nullptr);
}

// AF4-g64: the same kernel with the tensor maps of the prepared layout.
template <int MT, int NWC, int RPG>
__global__ void QG_XREG_BOUNDS gemv_xreg_af4_kernel(const Params p,
                                                    const __grid_constant__ CUtensorMap mq,
                                                    const __grid_constant__ CUtensorMap mm) {
    xreg_body<FMT_AF4, MT, NWC, RPG>(p, &mq, &mm);
}
#undef QG_XREG_BOUNDS

template <int FMT, int MT, int NWC, int RPG>
int launch(const DevCtx& dc, const Params& kp, int grid, int smem, bool pdl, cudaStream_t s) {
    auto kern = gemv_xreg_kernel<FMT, MT, NWC, RPG>;
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, kp);
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

constexpr int kRPG = 4;  // rows of a chunk per row group (per butterfly)

template <int FMT>
int dispatch(const DevCtx& dc, const Params& kp, int MT, int NWC, int grid, int smem, bool pdl,
             cudaStream_t s) {
    if (MT == 1) {
        if (NWC == 4) return launch<FMT, 1, 4, kRPG>(dc, kp, grid, smem, pdl, s);
        if (NWC == 8) return launch<FMT, 1, 8, kRPG>(dc, kp, grid, smem, pdl, s);
        if (NWC == 12) return launch<FMT, 1, 12, kRPG>(dc, kp, grid, smem, pdl, s);
        return launch<FMT, 1, 16, kRPG>(dc, kp, grid, smem, pdl, s);
    }
    if (MT == 2) {
        // Two input rows with sixteen consumer warps would spill: not planned.
        if (NWC == 4) return launch<FMT, 2, 4, kRPG>(dc, kp, grid, smem, pdl, s);
        if (NWC == 8) return launch<FMT, 2, 8, kRPG>(dc, kp, grid, smem, pdl, s);
        if (NWC == 12) return launch<FMT, 2, 12, kRPG>(dc, kp, grid, smem, pdl, s);
        return QG_ERR_UNSUPPORTED;
    }
    // Three or four input rows (128 registers of x per lane): four consumer
    // warps, one CTA per SM.
    if (NWC == 4) return launch<FMT, 4, 4, kRPG>(dc, kp, grid, smem, pdl, s);
    return QG_ERR_UNSUPPORTED;
}

}  // namespace xreg
}  // namespace qg
