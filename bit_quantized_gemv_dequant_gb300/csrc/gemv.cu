// GEMV / skinny-matmul dispatch (M <= 8 per launch; larger M is processed in
// slices of 8 rows of x): planning of the fast kernel of gemv_fast.cuh, the
// general kernel for shapes and alignments the fast one does not take, and
// the deterministic split-K finalization.
//
// Pages: fused_dual_proj_q4_0.rs (mlx-native 0.9.1), q4_k_gemv_v2.rs
// (ferrum-kernels 0.7.7), qmm_affine.rs (mlx-native 0.21.1).
//
// Split-K: when x for the M inputs does not fit in shared memory next to the
// weight stages (M*K*4 > 128 KB), the grid also splits K into KS slices. Each
// slice writes partial sums to the caller's workspace and splitk_finalize adds
// them in slice order, so results are deterministic and independent of the
// launch geometry.
#include <cuda_fp16.h>

#include <algorithm>

#include "gemv_fast.cuh"
#include "gemv_stream.cuh"
#include "gemv_xreg.cuh"
#include "qg_internal.cuh"

namespace qg {
namespace {

struct KParams {
    const uint8_t* w[2];
    float* out[2];
    const float* x;
    const float* s;
    const float* b;
    int M, N, K;
    int log2gs;
    int nw;
    long long q_row_bytes;
    int G;                    // groups per full row (affine)
};

// Sum of the KS slice partials in slice order: y = ((p0 + p1) + p2) + ...
__global__ void splitk_finalize(const float* __restrict__ partial, float* y0, float* y1, int nw,
                                int KS, long long MN) {
    const long long total = nw * MN;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int wi = (int)(i / MN);
        const long long o = i - wi * MN;
        float s = partial[((long long)wi) * MN + o];
        for (int ks = 1; ks < KS; ++ks) s += partial[((long long)ks * nw + wi) * MN + o];
        (wi == 0 ? y0 : y1)[o] = s;
    }
}

// ------------------------------------------------------------------ general
// Any shape and alignment the ABI accepts: one warp per (matrix, row), lanes
// stride along K decoding single elements straight from global memory.
template <int FMT>
__device__ __forceinline__ float weight_at(const uint8_t* row, int k, const float* srow,
                                           const float* brow, int log2gs) {
    if (FMT == FMT_Q4_0) {
        const uint8_t* blk = row + (k >> 5) * 18;
        const int j = k & 31;
        const uint8_t byte = blk[2 + (j & 15)];
        const int q = (j < 16) ? (byte & 15) : (byte >> 4);
        const float d = __half2float(__ushort_as_half((unsigned short)(blk[0] | (blk[1] << 8))));
        return __fmul_rn((float)(q - 8), d);
    } else if (FMT == FMT_Q4_K) {
        const uint8_t* blk = row + (k >> 8) * 144;
        const int within = k & 255, c = within >> 6, jj = within & 63, half = jj >> 5;
        const uint8_t byte = blk[16 + 32 * c + (jj & 31)];
        const int q = half ? (byte >> 4) : (byte & 15);
        const int j = 2 * c + half;
        const uint8_t* s12 = blk + 4;
        int sc, mn;
        if (j < 4) {
            sc = s12[j] & 63;
            mn = s12[j + 4] & 63;
        } else {
            sc = (s12[j + 4] & 15) | ((s12[j - 4] >> 6) << 4);
            mn = (s12[j + 4] >> 4) | ((s12[j] >> 6) << 4);
        }
        const float d = __half2float(__ushort_as_half((unsigned short)(blk[0] | (blk[1] << 8))));
        const float dmin =
            __half2float(__ushort_as_half((unsigned short)(blk[2] | (blk[3] << 8))));
        return __fmaf_rn(__fmul_rn(d, (float)sc), (float)q, -__fmul_rn(dmin, (float)mn));
    } else {
        int q;
        if (FMT == FMT_AFF_U8) {
            q = row[k];
        } else {
            const uint8_t byte = row[k >> 1];
            q = (k & 1) ? (byte >> 4) : (byte & 15);
        }
        return __fmaf_rn((float)q, srow[k >> log2gs], brow[k >> log2gs]);
    }
}

template <int FMT>
__global__ void __launch_bounds__(256) gemv_general_kernel(const KParams p) {
    const int warps = blockDim.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long rows_total = (long long)p.nw * p.N;
    for (long long gr = (long long)blockIdx.x * warps + (threadIdx.x >> 5); gr < rows_total;
         gr += (long long)gridDim.x * warps) {
        const int wi = (int)(gr / p.N);
        const int n = (int)(gr - (long long)wi * p.N);
        const uint8_t* row = p.w[wi] + (long long)n * p.q_row_bytes;
        const float* srow = p.s ? p.s + (long long)n * p.G : nullptr;
        const float* brow = p.b ? p.b + (long long)n * p.G : nullptr;
        for (int m0 = 0; m0 < p.M; m0 += 8) {
            const int mc = min(8, p.M - m0);
            float acc[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) acc[m] = 0.0f;
            for (int k = lane; k < p.K; k += 32) {
                const float w = weight_at<FMT>(row, k, srow, brow, p.log2gs);
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    if (m < mc) acc[m] = __fmaf_rn(w, p.x[(long long)(m0 + m) * p.K + k], acc[m]);
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1)
                    acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], off);
            }
            if (lane == 0)
                for (int m = 0; m < mc; ++m) p.out[wi][(long long)(m0 + m) * p.N + n] = acc[m];
        }
    }
}


// ------------------------------------------------------------------ planning
constexpr int kMaxStages = 32;
constexpr long long kXMaxBytes = 128 * 1024;

struct FmtGeo {
    int UE, unit_bytes, nh;
    bool sums;
};

FmtGeo geo(int fmt) {
    switch (fmt) {
        case FMT_Q4_0: return {32, 18, 1, false};
        case FMT_Q4_K: return {64, 36, 2, true};
        case FMT_AFF_U8: return {32, 32, 1, true};
        default: return {32, 16, 1, true};
    }
}

struct Plan {
    bool fast, co;
    int MT, R, GW, W, KS, klen, P, S, stage_bytes, q_stride, sb_stride, sb_off, xs_bytes,
        xsum_bytes, smem, grid_x, stages_per_w;
};

int ilog2(int v) {
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

long long row_bytes(int fmt, long long K) {
    switch (fmt) {
        case FMT_Q4_0: return K / 32 * 18;
        case FMT_Q4_K: return K / 256 * 144;
        case FMT_AFF_U8: return K;
        default: return K / 2;
    }
}

// Rows-per-stage options compiled for each M bucket (see fast::dispatch).
int r_options(int MT, int* out) {
    int n = 0;
    switch (MT) {
        case 1: out[n++] = 2; out[n++] = 4; out[n++] = 8; out[n++] = 16; break;
        case 2: out[n++] = 2; out[n++] = 4; break;
        case 4: out[n++] = 2; out[n++] = 4; break;
        default: out[n++] = 1; out[n++] = 2; out[n++] = 4; break;
    }
    return n;
}

// Planning of one launch for Mc (<= 8) input rows. A stage of R rows is one
// large TMA copy (bulk copies have a high per-copy cost, so pieces of >= 14 KB
// are preferred) shared by a group of GW warps, which split the k passes; GW
// depends only on the pass count, never on N or the number of matrices, so
// the arithmetic of every output is the same for single and dual calls. When
// the shared memory fits in half an SM, two CTAs (this kernel's and the next
// one's) can be resident together, which lets a programmatically launched
// successor stream its weights while this one drains.
Plan make_plan(const DevCtx& dc, const GemvArgs& a, int Mc) {
    Plan pl{};
    pl.fast = false;
    const bool affine = (a.fmt == FMT_AFF_U8 || a.fmt == FMT_AFF_PACKED);
    const FmtGeo g = geo(a.fmt);
    pl.MT = Mc <= 1 ? 1 : Mc <= 2 ? 2 : Mc <= 4 ? 4 : 8;
    pl.W = pl.MT <= 2 ? 16 : 12;
    // Q4_K with M bucket 8: eight consumer warps, one CTA per SM, so that a
    // stage can hold two rows (each x chunk then serves two rows).
    const bool q4k8 = a.fmt == FMT_Q4_K && pl.MT == 8;
    if (q4k8) pl.W = 8;
    // Eight consumer warps (two CTAs per SM: this launch's and the next one's)
    // when requested; M = 1 only.
    const bool w8 = pl.MT == 1 && launch_option(QG_OPT_STAGED_WARPS) == 8;
    if (w8) pl.W = 8;
    if (a.K % g.UE) return pl;
    for (int i = 0; i < a.nw; ++i)
        if (!aligned16(a.w[i])) return pl;
    if (row_bytes(a.fmt, a.K) % 16) return pl;
    if (affine) {
        if (a.gs < g.UE) return pl;  // a lane's unit must sit inside one group
        if ((a.K / a.gs) % 4 != 0 || !aligned16(a.scales) || !aligned16(a.biases)) return pl;
    }
    const int PASS = 32 * g.UE;
    // k-slices: x (padded to whole passes) and its sums must fit kXMaxBytes.
    int KS = 1;
    for (;; ++KS) {
        if (KS > 16) return pl;
        if (a.K % KS) continue;
        const long long klen = a.K / KS;
        if (klen % g.UE) continue;
        if (KS > 1 && (row_bytes(a.fmt, klen) % 16)) continue;
        if (affine && (klen % a.gs || (klen / a.gs) % 4)) continue;
        const long long P = (klen + PASS - 1) / PASS;
        const long long xb = (long long)pl.MT * P * PASS * 4 + (g.sums ? pl.MT * P * 32 * g.nh * 4 : 0);
        if (xb <= kXMaxBytes) break;
    }
    pl.KS = KS;
    pl.klen = (int)(a.K / KS);
    pl.P = (pl.klen + PASS - 1) / PASS;
    pl.GW = pl.P >= 4 ? 4 : (pl.P >= 2 ? 2 : 1);
    pl.q_stride = (int)row_bytes(a.fmt, pl.klen);
    pl.sb_stride = affine ? (pl.klen / a.gs) * 4 : 0;
    pl.xs_bytes = pl.MT * pl.P * PASS * 4;

    const int NG = pl.W / pl.GW;
    const int grid_cap = std::max(1, dc.num_sms / KS);
    const int co_budget = dc.smem_per_sm / 2 - dc.reserved_smem;  // two CTAs per SM
    int ropt[4];
    const int nr = r_options(pl.MT, ropt);
    bool have = false;
    long long best_key = -1;
    for (int ri = 0; ri < nr; ++ri) {
        const int R = ropt[ri];
        if (R > fast::max_rows(a.fmt, pl.MT, pl.W)) continue;
        if (w8 && R < 4) continue;
        const int V = pl.MT * R;
        const int sums = g.sums ? pl.MT * pl.P * 32 * g.nh : 0;
        for (int co = 1; co >= (w8 ? 1 : 0); --co) {
            if (co && q4k8) continue;  // its registers allow one CTA per SM
            const int stage = ((R * pl.q_stride + 2 * R * pl.sb_stride + 16) + 127) & ~127;
            const int budget = co ? co_budget : dc.max_smem_optin;
            // Per stage: the copy, two mbarriers, an arrival counter and the
            // group's partial sums (GW * V floats).
            const int per_stage = stage + 16 + 4 + (pl.GW > 1 ? pl.GW * V * 4 : 0);
            const int avail = budget - pl.xs_bytes - ((sums * 4 + 127) & ~127) - 128;
            if (avail <= 0) continue;
            int S = std::min(kMaxStages, avail / per_stage);
            if (S < 2) continue;
            if (S >= NG) S = NG * std::min(S / NG, 2);
            const int xsum_bytes =
                ((sums + S * (pl.GW > 1 ? pl.GW * V : 0) + S) * 4 + 127) & ~127;
            const long long spw = (a.N + R - 1) / R;
            const long long stages_total = spw * a.nw;
            const int grid = (int)std::min<long long>(stages_total, grid_cap);
            const double per_cta = (double)stages_total / grid;
            const int busy_groups = (int)std::min<double>(std::min(NG, S), std::ceil(per_cta));
            const int busy_warps = busy_groups * pl.GW;
            // Lexicographic preference (measured on GB300): most warps busy
            // (>= 3/4 of them), then more rows per stage (x reuse, fewer
            // per-stage costs), then two stages per group in flight, then
            // co-residency with the next kernel, then large copies.
            const long long key = ((long long)(busy_warps * 4 >= pl.W * 3) << 48) |
                                  ((long long)R << 40) | ((long long)(S >= 2 * NG) << 36) |
                                  ((long long)co << 32) | ((long long)(stage >= 14 * 1024) << 28) |
                                  ((long long)busy_warps << 16) | (long long)S;
            if (key > best_key) {
                best_key = key;
                have = true;
                pl.R = R;
                pl.S = S;
                pl.co = co != 0;
                pl.stage_bytes = stage;
                pl.xsum_bytes = xsum_bytes;
                pl.sb_off = R * pl.q_stride;
                pl.grid_x = grid;
                pl.stages_per_w = (int)spw;
            }
        }
    }
    if (!have) return pl;
    pl.smem = pl.xs_bytes + pl.xsum_bytes + pl.S * pl.stage_bytes + 2 * pl.S * 8;
    pl.fast = true;
    return pl;
}

// ----------------------------------------------------------- stream plan
// The streaming kernel (gemv_stream.cuh) for Mc <= 2: eligibility depends on
// the format, K, the group size and pointer alignment only, never on N or the
// number of matrices.
struct SPlan {
    bool ok;
    int MT, LPR, W, S, slot_bytes, sbl, xs_bytes, xsum_bytes, smem, grid, tpr, tasks_per_w;
};

SPlan make_stream_plan(const DevCtx& dc, const GemvArgs& a, int Mc, const float* x) {
    SPlan sp{};
    sp.ok = false;
    const long long mode = launch_option(QG_OPT_STREAM);
    if (Mc > 2 || mode == 0) return sp;
    // Automatic: where it measured faster than the staged kernel on GB300:
    // Q4_K, except two input rows with K above 8192 (FFN down, K = 12288:
    // 21.4 us against 19.4 us). 2 takes it for every eligible call. The
    // choice depends on the format, the rows and K only, never on N.
    if (mode == 1 && (a.fmt != FMT_Q4_K || (Mc == 2 && a.K > 8192))) return sp;
    const bool affine = (a.fmt == FMT_AFF_U8 || a.fmt == FMT_AFF_PACKED);
    if (a.K % 256) return sp;
    const long long U = a.K / 256;
    int LPR = 1;
    while (LPR < 32 && U % (2 * LPR) == 0) LPR *= 2;
    if (LPR < 4) return sp;
    for (int i = 0; i < a.nw; ++i)
        if (!aligned16(a.w[i])) return sp;
    if (!aligned16(x)) return sp;
    if (affine && (a.gs < 32 || !aligned16(a.scales) || !aligned16(a.biases))) return sp;
    const int RW = 32 / LPR;
    const long long rb = row_bytes(a.fmt, a.K);
    if (rb * RW >= (1ll << 31) || a.K > (1 << 24)) return sp;
    sp.MT = Mc;
    sp.LPR = LPR;
    sp.tpr = (int)(U / LPR);
    sp.tasks_per_w = (int)((a.N + RW - 1) / RW);
    const bool sums = a.fmt != FMT_Q4_0;
    sp.xs_bytes = (int)(sp.MT * U * 65 * 16);            // 64 float4 + 1 padding per unit
    sp.xsum_bytes = sums ? (int)(sp.MT * U * 12 * 4) : 0;  // 8 sums + 4 padding per unit
    const int UB = a.fmt == FMT_AFF_U8 ? 256 : a.fmt == FMT_AFF_PACKED ? 128 : 144;
    sp.sbl = affine ? (a.gs == 32 ? 32 : 16) : 0;
    sp.slot_bytes = 32 * UB + 64 * sp.sbl;
    const long long fixed = (long long)sp.xs_bytes + sp.xsum_bytes + 128;
    auto smem_of = [&](int W, int S) { return fixed + (long long)W * S * sp.slot_bytes; };
    const long long co_budget = dc.smem_per_sm / 2 - dc.reserved_smem;
    const int ow = (int)launch_option(QG_OPT_STREAM_WARPS), os = (int)launch_option(QG_OPT_STREAM_SLOTS);
    int W = 0, S = 0;
    if (ow > 0 || os > 0) {
        const int w = ow > 0 ? ow : 8, s2 = os > 0 ? os : 2;
        if (smem_of(w, s2) <= dc.max_smem_optin) {
            W = w;
            S = s2;
        }
    }
    if (W == 0) {
        // Two CTAs per SM when 8 warps with two slots each fit in half an SM;
        // otherwise one CTA with the most slots (up to 4) that fit.
        if (smem_of(8, 2) <= co_budget) {
            W = 8;
            S = 2;
        } else {
            for (int s2 = 4; s2 >= 2 && W == 0; --s2)
                if (smem_of(8, s2) <= dc.max_smem_optin) {
                    W = 8;
                    S = s2;
                }
            for (int w = 4; w >= 1 && W == 0; w /= 2)
                if (smem_of(w, 2) <= dc.max_smem_optin) {
                    W = w;
                    S = 2;
                }
        }
    }
    if (W == 0) return sp;
    sp.W = W;
    sp.S = S;
    sp.smem = (int)smem_of(W, S);
    // Two CTAs per SM when they fit (both of this launch; as they retire, the
    // next launch's CTAs take their place and start streaming).
    const long long total = (long long)sp.tasks_per_w * a.nw;
    const int per_sm = (sp.smem + dc.reserved_smem) * 2 <= dc.smem_per_sm ? 2 : 1;
    sp.grid = (int)std::min<long long>(total, (long long)per_sm * dc.num_sms);
    sp.ok = true;
    return sp;
}

// ------------------------------------------------------------ xreg plan
// The register-resident-x kernel (gemv_xreg.cuh) for Mc <= 2. Its geometry
// (warps per row group, consumer warps, rows per chunk) depends on the format
// and K only, never on N or the number of matrices.
struct XPlan {
    bool ok;
    int NWC, WG, NRG, RC, S, slot_bytes, sb_off, smem, grid, units, rbuf, red_floats;
};

XPlan make_xreg_plan(const DevCtx& dc, const GemvArgs& a, int Mc, const float* x) {
    XPlan xp{};
    xp.ok = false;
    if (Mc > 4 || launch_option(QG_OPT_XREG) == 0) return xp;
    const int MT = Mc <= 2 ? Mc : 4;  // three rows run as four (one of zeros)
    const bool affine = (a.fmt == FMT_AFF_U8 || a.fmt == FMT_AFF_PACKED);
    if (a.K % 32 || a.K > 16384) return xp;
    const long long units = a.K / 32;
    long long WG;
    if (a.fmt == FMT_Q4_0) {
        if (a.K % 256) return xp;          // 16-byte aligned rows
        WG = 2 * ((units + 63) / 64);      // warps of one block parity each
    } else {
        if (affine && (a.gs < 32 || (a.K / a.gs) % 4)) return xp;
        WG = (units + 31) / 32;
    }
    if (WG > 16) return xp;
    for (int i = 0; i < a.nw; ++i)
        if (!aligned16(a.w[i])) return xp;
    if (!aligned16(x)) return xp;
    if (affine && (!aligned16(a.scales) || !aligned16(a.biases))) return xp;
    if ((long long)a.nw * a.N >= (1ll << 31)) return xp;
    if (MT == 4 && (WG > 4 || 4 % WG)) return xp;  // four x rows: only four consumer warps fit
    // Four rows of x at once (one CTA of four consumer warps per SM) measured
    // faster than the staged kernel for Q4_K and affine weights (M = 4 / 8:
    // Q4_K 22.0 / 43.9 us against 24.3 / 47.4 us at N = 12288; affine u8
    // 19.2 against 22.9 us at M = 8) but slower for Q4_0 (dual M = 4:
    // 15.5 against 13.8 us), which keeps the staged kernel.
    if (MT == 4 && a.fmt == FMT_Q4_0) return xp;
    int NWC = (8 % WG == 0) ? 8 : (12 % WG == 0) ? 12 : 16;
    // Four consumer warps (four CTAs, i.e. four calls, per SM) when calls are
    // declared independent (QG_OPT_PDL = 2): consecutive calls then overlap,
    // and more of them in flight hide each CTA's start-up and tail. A call
    // that waits for its predecessor computes alone, and does better with
    // eight warps (two CTAs per SM: this call's and the next one's). A call
    // that runs alone keeps eight (measured against four and sixteen for the
    // dual N = K = 4096 call: 17.2 us per host round trip against 18.8 and
    // 18.0) and takes all of the SM's shared memory.
    const long long want_w = launch_option(QG_OPT_XREG_WARPS);
    if (MT == 4) {
        NWC = 4;
    } else if (want_w != 0) {
        // A requested count that the row groups do not divide, or sixteen
        // warps with two x rows (more registers than 17 warps allow), falls
        // back to the automatic choice.
        if (want_w % WG == 0 && !(want_w == 16 && MT == 2)) NWC = (int)want_w;
    } else if (!a.isolated && WG <= 4 && 4 % WG == 0 && launch_option(QG_OPT_PDL) == 2) {
        NWC = 4;
    }
    if (NWC == 16 && MT == 2) return xp;  // two x rows need more registers than 17 warps allow
    const int NRG = std::min<int>(8, NWC / (int)WG);
    const int RC = NRG * xreg::kRPG;
    const long long rb = row_bytes(a.fmt, a.K);
    const int G = affine ? (int)(a.K / a.gs) : 0;
    const long long slot = ((RC * rb + (affine ? 2ll * RC * G * 4 : 0)) + 127) & ~127ll;
    // Packed and one-code-per-byte affine calls must take the same kernel
    // (their results are bitwise equal only then): whether the plan fits is
    // decided on the larger, one-code-per-byte slot for both.
    const long long slot_fit = affine ? ((RC * a.K + 2ll * RC * G * 4) + 127) & ~127ll : slot;
    // CTAs per call. For calls with one or two rows of x declared
    // independent (QG_OPT_PDL = 2), whose CTAs run beside those of the calls
    // around them, fewer, longer CTAs spend less per call on start-up and x
    // staging: three per four SMs for one row of x on four warps, one per two
    // SMs for one row on more warps, one per four SMs for two rows. Measured
    // over runs of hundreds of calls (us per call, one per SM / three per
    // four / one per two / one per four): dual N = K = 4096 3.83 / 3.61 /
    // 3.55 / 4.03, Q4_K N = 12288 6.63 / 6.42 / 6.48 / 7.54, decode layer
    // 22.2 / 21.0 / 21.5 / 20.5; two rows: K+V 2.37 / 2.07 / 1.76 / 1.67, Q4_K
    // K = 12288 14.9 / - / 12.1 / 9.8, decode layer 33.6 / - / 29.5 / 28.2;
    // over 20 calls, where the longer CTAs' fill and drain count, the dual
    // call 4.36-4.46 / 4.36 / 4.46 / 5.28. One per SM for a call that waits for
    // its predecessor or runs alone, and for four rows of x, whose calls run
    // beside the staged kernel's single wave of CTAs (halving them made the
    // M = 4 decode layer 93 us against 74: the staged CTAs waited for the
    // longer ones to leave their SMs).
    const bool shares_sm = ((NWC == 8 || NWC == 12) && MT == 1) || (NWC == 4 && MT <= 2);
    const long long ctas_opt = launch_option(QG_OPT_XREG_CTAS);
    const bool overlapped =
        MT <= 2 && !a.isolated && !a.x_from_prev && launch_option(QG_OPT_PDL) == 2;
    const long long quarters = MT == 2 ? 1 : NWC == 4 ? 3 : 2;  // SMs per call, in quarters
    const long long grid_max = ctas_opt > 0 ? (long long)dc.num_sms * ctas_opt
                               : overlapped ? std::max<long long>(1, dc.num_sms * quarters / 4)
                                            : (long long)dc.num_sms;
    const long long rows_cta = ((long long)a.nw * a.N + grid_max - 1) / grid_max;
    // Rows of per-warp partial sums buffered before a flush: the CTA's whole
    // share when it fits in 16 KB, and never fewer than one chunk.
    const long long rbuf = std::max<long long>(RC, std::min<long long>(rows_cta, 4096 / (MT * WG)));
    const long long per_slot = slot + 16;
    // Partial sums, then the staging area of x (MT * K floats).
    const long long red_floats = (rbuf * MT * WG + 3) & ~3ll;
    const long long fixed = (red_floats + (long long)MT * a.K) * 4 + (long long)NWC * MT * 4 + 128;
    // Eight or twelve consumer warps with one input row fit twice on an SM
    // (this call's CTA and the next one's), four consumer warps four times
    // (three times with two input rows); otherwise one CTA per SM.
    const bool co = !a.isolated && shares_sm;
    const int per_sm = NWC == 4 ? (MT == 1 ? 4 : 3) : 2;
    long long budget = co ? (long long)dc.smem_per_sm / per_sm - dc.reserved_smem : dc.max_smem_optin;
    long long S = std::min<long long>(16, (budget - fixed) / per_slot);
    if ((budget - fixed) / (slot_fit + 16) < 2) {
        budget = dc.max_smem_optin;
        S = std::min<long long>(16, (budget - fixed) / per_slot);
    }
    if ((budget - fixed) / (slot_fit + 16) < 2) return xp;
    xp.NWC = NWC;
    xp.WG = (int)WG;
    xp.NRG = NRG;
    xp.RC = RC;
    xp.S = (int)S;
    xp.slot_bytes = (int)slot;
    xp.sb_off = (int)(RC * rb);
    xp.smem = (int)(S * per_slot + fixed - 128);
    xp.grid = (int)std::min<long long>((long long)a.nw * a.N, grid_max);
    xp.units = (int)units;
    xp.rbuf = (int)rbuf;
    xp.red_floats = (int)red_floats;
    xp.ok = true;
    return xp;
}

template <int FMT>
int launch_general(const DevCtx& dc, const KParams& kp, cudaStream_t s) {
    const long long rows = (long long)kp.nw * kp.N;
    const long long blocks = std::min<long long>((rows + 7) / 8, (long long)dc.num_sms * 16);
    gemv_general_kernel<FMT><<<(int)blocks, 256, 0, s>>>(kp);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

}  // namespace

int stream_launch_q4_0(const DevCtx&, const stream::Params&, int, int, int, int, int, bool, cudaStream_t);
int stream_launch_q4_k(const DevCtx&, const stream::Params&, int, int, int, int, int, bool, cudaStream_t);
int stream_launch_aff_u8(const DevCtx&, const stream::Params&, int, int, int, int, int, bool,
                         cudaStream_t);
int stream_launch_aff_packed(const DevCtx&, const stream::Params&, int, int, int, int, int, bool,
                             cudaStream_t);
int xreg_launch_q4_0(const DevCtx&, const xreg::Params&, int, int, int, int, bool, cudaStream_t);
int xreg_launch_q4_k(const DevCtx&, const xreg::Params&, int, int, int, int, bool, cudaStream_t);
int xreg_launch_aff_u8(const DevCtx&, const xreg::Params&, int, int, int, int, bool, cudaStream_t);
int xreg_launch_aff_packed(const DevCtx&, const xreg::Params&, int, int, int, int, bool,
                           cudaStream_t);
int fast_launch_q4_0(const DevCtx&, const fast::Params&, int, int, int, int, int, int, bool,
                      cudaStream_t);
int fast_launch_q4_k(const DevCtx&, const fast::Params&, int, int, int, int, int, int, bool,
                      cudaStream_t);
int fast_launch_aff_u8(const DevCtx&, const fast::Params&, int, int, int, int, int, int, bool,
                      cudaStream_t);
int fast_launch_aff_packed(const DevCtx&, const fast::Params&, int, int, int, int, int, int,
                           bool, cudaStream_t);

// Calls with more than two rows of x run in slices of four on the
// register-resident-x kernel when it takes four rows for this shape (no
// workspace), else in slices of eight on the staged kernel.
bool xreg_four_row_slices(const DevCtx& dc, const GemvArgs& a) {
    return a.M >= 3 && make_xreg_plan(dc, a, 4, a.x).ok;
}

// Every slice of the call runs on the register-resident-x kernel. That
// kernel reads x with plain loads and writes y with plain stores and needs
// no workspace, so x and y may then live in mapped host memory.
bool gemv_xreg_only(const DevCtx& dc, const GemvArgs& a) {
    const int step = xreg_four_row_slices(dc, a) ? 4 : 8;
    for (long long m0 = 0; m0 < a.M; m0 += step) {
        const int Mc = (int)std::min<long long>(step, a.M - m0);
        if (!make_xreg_plan(dc, a, Mc, a.x + m0 * a.K).ok) return false;
    }
    return true;
}

size_t gemv_workspace_bytes(const DevCtx& dc, const GemvArgs& a) {
    if (xreg_four_row_slices(dc, a)) return 0;
    size_t worst = 0;
    for (long long m0 = 0; m0 < a.M; m0 += 8) {
        const int Mc = (int)std::min<long long>(8, a.M - m0);
        const Plan pl = make_plan(dc, a, Mc);
        if (pl.fast && pl.KS > 1)
            worst = std::max(worst, (size_t)pl.KS * a.nw * Mc * (size_t)a.N * sizeof(float));
    }
    return worst;
}

int gemv_launch(const DevCtx& dc, const GemvArgs& a, void* ws, size_t ws_bytes, cudaStream_t s) {
    const bool affine = (a.fmt == FMT_AFF_U8 || a.fmt == FMT_AFF_PACKED);
    const int step = xreg_four_row_slices(dc, a) ? 4 : 8;
    for (long long m0 = 0; m0 < a.M; m0 += step) {
        const int Mc = (int)std::min<long long>(step, a.M - m0);
        const float* x = a.x + m0 * a.K;
        float* y0 = a.y[0] + m0 * a.N;
        float* y1 = (a.nw > 1 ? a.y[1] : a.y[0]) + m0 * a.N;
        int rc;
        const XPlan xp = make_xreg_plan(dc, a, Mc, x);
        if (xp.ok) {
            xreg::Params kp{};
            kp.w[0] = a.w[0];
            kp.w[1] = a.nw > 1 ? a.w[1] : a.w[0];
            kp.out[0] = y0;
            kp.out[1] = y1;
            kp.x = x;
            kp.s = a.scales;
            kp.b = a.biases;
            kp.M = Mc;
            kp.N = (int)a.N;
            kp.K = (int)a.K;
            kp.nw = a.nw;
            kp.log2gs = affine ? ilog2(a.gs) : 0;
            kp.G = affine ? (int)(a.K / a.gs) : 0;
            kp.row_bytes = (int)row_bytes(a.fmt, a.K);
            const int rows_total = (int)(a.nw * a.N);
            kp.rows_base = rows_total / xp.grid;
            kp.rows_rem = rows_total % xp.grid;
            kp.S = xp.S;
            kp.slot_bytes = xp.slot_bytes;
            kp.sb_off = xp.sb_off;
            kp.WG = xp.WG;
            kp.NRG = xp.NRG;
            kp.RC = xp.RC;
            kp.units = xp.units;
            kp.rbuf = xp.rbuf;
            kp.red_floats = xp.red_floats;
            kp.ahead = (int)std::min<long long>(launch_option(QG_OPT_XREG_AHEAD), xp.S);
            kp.err = dc.err;
            const long long pdl_mode = a.x_from_prev ? 1 : launch_option(QG_OPT_PDL);
            const bool pdl = pdl_mode != 0;
            kp.dep_wait = pdl_mode == 2 ? 0 : 1;
            const int MT = Mc <= 2 ? Mc : 4;
            switch (a.fmt) {
                case FMT_Q4_0:
                    rc = xreg_launch_q4_0(dc, kp, MT, xp.NWC, xp.grid, xp.smem, pdl, s);
                    break;
                case FMT_Q4_K:
                    rc = xreg_launch_q4_k(dc, kp, MT, xp.NWC, xp.grid, xp.smem, pdl, s);
                    break;
                case FMT_AFF_U8:
                    rc = xreg_launch_aff_u8(dc, kp, MT, xp.NWC, xp.grid, xp.smem, pdl, s);
                    break;
                default:
                    rc = xreg_launch_aff_packed(dc, kp, MT, xp.NWC, xp.grid, xp.smem, pdl, s);
                    break;
            }
            if (rc != QG_OK) return rc;
            continue;
        }
        const SPlan sp = make_stream_plan(dc, a, Mc, x);
        if (sp.ok) {
            stream::Params kp{};
            kp.w[0] = a.w[0];
            kp.w[1] = a.nw > 1 ? a.w[1] : a.w[0];
            kp.out[0] = y0;
            kp.out[1] = y1;
            kp.x = x;
            kp.s = a.scales;
            kp.b = a.biases;
            kp.M = Mc;
            kp.N = (int)a.N;
            kp.K = (int)a.K;
            kp.nw = a.nw;
            kp.tpr = sp.tpr;
            kp.tpr_magic = sp.tpr > 1 ? (uint32_t)(((1ull << 32) + sp.tpr - 1) / sp.tpr) : 0u;
            kp.tasks_per_w = sp.tasks_per_w;
            kp.total_tasks = sp.tasks_per_w * a.nw;
            kp.tasks_base = kp.total_tasks / sp.grid;
            kp.tasks_rem = kp.total_tasks % sp.grid;
            kp.S = sp.S;
            kp.slot_bytes = sp.slot_bytes;
            kp.sbl = sp.sbl;
            kp.log2gs = affine ? ilog2(a.gs) : 0;
            kp.G = affine ? (int)(a.K / a.gs) : 0;
            kp.row_bytes = row_bytes(a.fmt, a.K);
            kp.xs_bytes = sp.xs_bytes;
            kp.xsum_bytes = sp.xsum_bytes;
            kp.zero = 0u;
            const bool pdl = launch_option(QG_OPT_PDL) != 0;
            switch (a.fmt) {
                case FMT_Q4_0:
                    rc = stream_launch_q4_0(dc, kp, sp.MT, sp.LPR, sp.grid, sp.W, sp.smem, pdl, s);
                    break;
                case FMT_Q4_K:
                    rc = stream_launch_q4_k(dc, kp, sp.MT, sp.LPR, sp.grid, sp.W, sp.smem, pdl, s);
                    break;
                case FMT_AFF_U8:
                    rc = stream_launch_aff_u8(dc, kp, sp.MT, sp.LPR, sp.grid, sp.W, sp.smem, pdl, s);
                    break;
                default:
                    rc = stream_launch_aff_packed(dc, kp, sp.MT, sp.LPR, sp.grid, sp.W, sp.smem, pdl, s);
                    break;
            }
            if (rc != QG_OK) return rc;
            continue;
        }
        const Plan pl = make_plan(dc, a, Mc);
        if (!pl.fast) {
            KParams kp{};
            kp.w[0] = a.w[0];
            kp.w[1] = a.nw > 1 ? a.w[1] : a.w[0];
            kp.out[0] = y0;
            kp.out[1] = y1;
            kp.x = x;
            kp.s = a.scales;
            kp.b = a.biases;
            kp.M = Mc;
            kp.N = (int)a.N;
            kp.K = (int)a.K;
            kp.nw = a.nw;
            kp.log2gs = affine ? ilog2(a.gs) : 0;
            kp.G = affine ? (int)(a.K / a.gs) : 0;
            kp.q_row_bytes = row_bytes(a.fmt, a.K);
            switch (a.fmt) {
                case FMT_Q4_0: rc = launch_general<FMT_Q4_0>(dc, kp, s); break;
                case FMT_Q4_K: rc = launch_general<FMT_Q4_K>(dc, kp, s); break;
                case FMT_AFF_U8: rc = launch_general<FMT_AFF_U8>(dc, kp, s); break;
                default: rc = launch_general<FMT_AFF_PACKED>(dc, kp, s); break;
            }
            if (rc != QG_OK) return rc;
            continue;
        }
        fast::Params kp{};
        kp.w[0] = a.w[0];
        kp.w[1] = a.nw > 1 ? a.w[1] : a.w[0];
        kp.out[0] = y0;
        kp.out[1] = y1;
        kp.x = x;
        kp.s = a.scales;
        kp.b = a.biases;
        kp.M = Mc;
        kp.N = (int)a.N;
        kp.K = (int)a.K;
        kp.log2gs = affine ? ilog2(a.gs) : 0;
        kp.nw = a.nw;
        kp.klen = pl.klen;
        kp.P = pl.P;
        kp.units = pl.klen / geo(a.fmt).UE;
        kp.chunks_per_w = pl.stages_per_w;
        kp.total_chunks = pl.stages_per_w * a.nw;
        kp.chunk_base = kp.total_chunks / pl.grid_x;
        kp.chunk_rem = kp.total_chunks % pl.grid_x;
        // The in-flight limit helps the bandwidth-bound M <= 2 calls; the
        // compute-bound M >= 4 ones keep every stage in flight.
        kp.ahead = pl.MT <= 2 ? std::min<int>((int)launch_option(QG_OPT_STAGES_AHEAD), pl.S) : 0;
        kp.S = pl.S;
        kp.stage_bytes = pl.stage_bytes;
        kp.q_stride = pl.q_stride;
        kp.sb_stride = pl.sb_stride;
        kp.sb_off = pl.sb_off;
        kp.q_row_bytes = row_bytes(a.fmt, a.K);
        kp.G = affine ? (int)(a.K / a.gs) : 0;
        kp.KS = pl.KS;
        kp.xs_bytes = pl.xs_bytes;
        kp.xsum_bytes = pl.xsum_bytes;
        kp.magic = 0x4B000000u;
        kp.err = dc.err;
        // Independent calls (QG_OPT_PDL = 2) need not wait for their
        // predecessor, except when split-K partials go to a workspace that
        // consecutive calls may share.
        kp.dep_wait = (launch_option(QG_OPT_PDL) == 2 && !a.x_from_prev && pl.KS == 1) ? 0 : 1;
        if (pl.KS > 1) {
            const size_t need = (size_t)pl.KS * a.nw * Mc * (size_t)a.N * sizeof(float);
            if (!ws || ws_bytes < need) return QG_ERR_WORKSPACE;
            kp.partial = static_cast<float*>(ws);
        }
        const bool pdl = launch_option(QG_OPT_PDL) != 0;
        switch (a.fmt) {
            case FMT_Q4_0:
                rc = fast_launch_q4_0(dc, kp, pl.MT, pl.R, pl.GW, pl.W, pl.grid_x, pl.smem, pdl, s);
                break;
            case FMT_Q4_K:
                rc = fast_launch_q4_k(dc, kp, pl.MT, pl.R, pl.GW, pl.W, pl.grid_x, pl.smem, pdl, s);
                break;
            case FMT_AFF_U8:
                rc = fast_launch_aff_u8(dc, kp, pl.MT, pl.R, pl.GW, pl.W, pl.grid_x, pl.smem, pdl, s);
                break;
            default:
                rc = fast_launch_aff_packed(dc, kp, pl.MT, pl.R, pl.GW, pl.W, pl.grid_x, pl.smem, pdl, s);
                break;
        }
        if (rc != QG_OK) return rc;
        if (pl.KS > 1) {
            const long long MN = (long long)Mc * a.N;
            const long long blocks = std::min<long long>((a.nw * MN + 255) / 256, dc.num_sms * 8);
            splitk_finalize<<<(int)blocks, 256, 0, s>>>(kp.partial, y0, y1, a.nw, pl.KS, MN);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return cuda_fail(e);
        }
    }
    return QG_OK;
}

}  // namespace qg
