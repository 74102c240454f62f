// Dequantize-fused GEMV / skinny matmul on CUDA cores (M <= 8 per launch).
//
// Pages: fused_dual_proj_q4_0.rs (mlx-native 0.9.1), q4_k_gemv_v2.rs
// (ferrum-kernels 0.7.7) and qmm_affine.rs (mlx-native 0.21.1) define the
// operations and their host contracts; their Metal kernels (64-thread
// threadgroups, two rows per simdgroup) are not reused. This design is
// written for sm_103a:
//
//  * One persistent CTA per SM (8 consumer warps + 1 producer warp). The CTAs
//    split the list of row chunks (R consecutive rows of one weight matrix)
//    into contiguous, balanced ranges.
//  * The producer streams each chunk's bytes from HBM into a ring of shared
//    memory stages with 1-D TMA bulk copies (cp.async.bulk, evict-first L2
//    policy) completing on mbarriers, so a whole SM's share of the weights
//    can be in flight at once without holding registers.
//  * x (one k-slice of it) is staged once per CTA in shared memory, permuted
//    so that each lane's 8 inputs for a 256-element pass are two conflict-free
//    float4 loads. A warp loads them into registers once per pass and reuses
//    them for the R rows of its chunk and all M inputs.
//  * Nibbles become exact floats with an exponent-bias trick (OR into the
//    mantissa of 2^23, subtract), are multiplied by x in f32, and the per-
//    block scale is applied once per lane-block. Partial sums of the R*M
//    outputs are reduced across the warp with a transposing butterfly.
//  * When x does not fit (M*K*4 > 128 KB) the grid also splits K into KS
//    slices; each slice writes partial sums to the workspace and a second
//    kernel adds them in slice order, so results stay deterministic.
//
// Every output's arithmetic depends only on (format, M bucket, K, KS), never
// on which CTA, warp or chunk computed it, so the dual projection is bitwise
// equal to two single projections.
#include <cuda_fp16.h>

#include <algorithm>

#include "qg_internal.cuh"

namespace qg {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;
constexpr int kPass = 256;            // K elements per lane-pass (32 lanes x 8)
constexpr int kMaxStages = 24;
constexpr size_t kXMaxBytes = 128 * 1024;

struct KParams {
    const uint8_t* w[2];
    float* out[2];            // y (KS == 1) or unused (KS > 1: partial)
    float* partial;           // [KS][nw][M][N] when KS > 1
    const float* x;
    const float* s;
    const float* b;
    int M, N, K;
    int log2gs;
    int nw;
    int klen, passes;
    int chunks_per_w, total_chunks;
    int S, stage_bytes;
    int q_stride, sb_stride, sb_off;
    long long q_row_bytes;
    int G;                    // groups per full row (affine)
    int KS;
    unsigned* err;
};

__host__ __device__ constexpr int q_bytes_per_pass(int fmt) {
    return fmt == FMT_AFF_U8 ? 256 : (fmt == FMT_AFF_PACKED ? 128 : 144);
}

// Exact float of a small code q (< 2^23): 2^23 + q, minus 2^23 (+ bias).
__device__ __forceinline__ float code_f(uint32_t q) {
    return __int_as_float(0x4B000000u | q) - 8388608.0f;
}
__device__ __forceinline__ float code_f_minus8(uint32_t q) {
    return __int_as_float(0x4B000000u | q) - 8388616.0f;
}

// Position in the permuted x layout of element e (0 <= e < klen) of input m:
// [m][pass][plane][lane][4]; each lane reads its 8 values as two float4.
template <int FMT>
__device__ __forceinline__ int x_index(int m, int e, int passes) {
    const int pp = e >> 8, ee = e & 255;
    int plane, lane, t;
    if (FMT == FMT_Q4_0) {
        const int j = ee & 31;
        plane = j >> 4;
        lane = (ee >> 5) * 4 + ((j & 15) >> 2);
        t = j & 3;
    } else if (FMT == FMT_Q4_K) {
        const int j = ee & 63;
        plane = j >> 5;
        lane = (ee >> 6) * 8 + ((j & 31) >> 2);
        t = j & 3;
    } else {
        lane = ee >> 3;
        plane = (ee >> 2) & 1;
        t = ee & 3;
    }
    return (((m * passes + pp) * 2 + plane) * 32 + lane) * 4 + t;
}

// The (scale, min) 6-bit pair of sub-block j from the 12 packed bytes held
// as three little-endian words.
__device__ __forceinline__ void q4k_pair(uint32_t s0, uint32_t s1, uint32_t s2, int j, int& sc,
                                         int& mn) {
    const int jj = j & 3, sh = 8 * jj;
    const uint32_t b0 = (s0 >> sh) & 0xFF, b1 = (s1 >> sh) & 0xFF, b2 = (s2 >> sh) & 0xFF;
    if (j < 4) {
        sc = b0 & 63;
        mn = b1 & 63;
    } else {
        sc = (b2 & 15) | ((b0 >> 6) << 4);
        mn = (b2 >> 4) | ((b1 >> 6) << 4);
    }
}

// Warp reduction of V values at once. Afterwards lane l holds the full sum
// of value l / (32 / V). Each value is summed over the same xor-butterfly
// tree as a plain one-value reduction.
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

template <int FMT, int MT, int R>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const KParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    float* xs = reinterpret_cast<float*>(smem);
    const int x_bytes = (MT * p.klen * 4 + 127) & ~127;
    uint8_t* stages = smem + x_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(stages + (size_t)p.S * p.stage_bytes);
    uint64_t* empty = full + p.S;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ks = blockIdx.y;
    const int k0 = ks * p.klen;
    const int c_begin = (int)((long long)p.total_chunks * blockIdx.x / gridDim.x);
    const int c_end = (int)((long long)p.total_chunks * (blockIdx.x + 1) / gridDim.x);
    const int n_local = c_end - c_begin;
    constexpr bool kAffine = (FMT == FMT_AFF_U8 || FMT == FMT_AFF_PACKED);

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.S; ++i) {
            mbar_init(smem_addr(&full[i]), 1);
            mbar_init(smem_addr(&empty[i]), 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    // ------------------------------------------------------------ producer
    if (warp == kConsumerWarps) {
        if (lane != 0) return;
        const uint64_t pol = l2_evict_first();
        const long long q_off = (long long)(k0 / kPass) * q_bytes_per_pass(FMT);
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
            const int cid = c_begin + i;
            const int wi = cid / p.chunks_per_w;
            const int row0 = (cid - wi * p.chunks_per_w) * R;
            const int rows = min(R, p.N - row0);
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
                    bulk_g2s(smem_addr(dst + p.sb_off + R * p.sb_stride),
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
                        bulk_g2s(smem_addr(dst + p.sb_off + (R + r) * p.sb_stride), p.b + go,
                                 p.sb_stride, bar, pol);
                    }
                }
            }
            issued = i + 1;
        }
        if (!ok) {
            // Wait (bounded) for every stage's most recent copies to land
            // before this block's shared memory can be released.
            for (int st = 0; st < p.S && st < issued; ++st) {
                const int last = st + ((issued - 1 - st) / p.S) * p.S;
                if (!mbar_wait(smem_addr(&full[st]), (last / p.S) & 1))
                    report_error(p.err, DEVERR_WAIT_DRAIN);
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    for (int idx = threadIdx.x; idx < MT * p.klen; idx += kConsumerThreads) {
        const int m = idx / p.klen, e = idx - m * p.klen;
        const float v = (m < p.M) ? p.x[(long long)m * p.K + k0 + e] : 0.0f;
        xs[x_index<FMT>(m, e, p.passes)] = v;
    }
    named_bar_sync(1, kConsumerThreads);

    // Lane-constant parts of the decode.
    int q4k_j0 = 0;
    if (FMT == FMT_Q4_K) q4k_j0 = 2 * (lane >> 3);

    for (int i = warp; i < n_local; i += kConsumerWarps) {
        const int st = i % p.S, use = i / p.S;
        if (!mbar_wait(smem_addr(&full[st]), use & 1)) {
            report_error(p.err, DEVERR_WAIT_FULL);
            return;
        }
        const int cid = c_begin + i;
        const int wi = cid / p.chunks_per_w;
        const int row0 = (cid - wi * p.chunks_per_w) * R;
        const int rows = min(R, p.N - row0);
        const uint8_t* stg = stages + (size_t)st * p.stage_bytes;

        float acc[MT][R];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < R; ++r) acc[m][r] = 0.0f;

#pragma unroll 1
        for (int pp = 0; pp < p.passes; ++pp) {
            float xl[MT][4], xh[MT][4];
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float4 a = *reinterpret_cast<const float4*>(
                    xs + (((m * p.passes + pp) * 2 + 0) * 32 + lane) * 4);
                const float4 c = *reinterpret_cast<const float4*>(
                    xs + (((m * p.passes + pp) * 2 + 1) * 32 + lane) * 4);
                xl[m][0] = a.x; xl[m][1] = a.y; xl[m][2] = a.z; xl[m][3] = a.w;
                xh[m][0] = c.x; xh[m][1] = c.y; xh[m][2] = c.z; xh[m][3] = c.w;
            }
            float sxl[MT], sxh[MT];
            if (FMT != FMT_Q4_0) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    sxl[m] = (xl[m][0] + xl[m][1]) + (xl[m][2] + xl[m][3]);
                    sxh[m] = (xh[m][0] + xh[m][1]) + (xh[m][2] + xh[m][3]);
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (r >= rows) break;
                const uint8_t* row = stg + r * p.q_stride;
                if (FMT == FMT_Q4_0) {
                    const int bl = pp * 8 + (lane >> 2);
                    const int off = bl * 18 + 2 + (lane & 3) * 4;
                    const uint32_t* rw = reinterpret_cast<const uint32_t*>(row);
                    const uint32_t lo = rw[off >> 2], hi = rw[(off >> 2) + 1];
                    const uint32_t v = __funnelshift_r(lo, hi, (off & 3) * 8);
                    const float d =
                        __half2float(*reinterpret_cast<const __half*>(row + bl * 18));
                    float f[8];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        f[t] = code_f_minus8((v >> (8 * t)) & 0xF);
                        f[4 + t] = code_f_minus8((v >> (8 * t + 4)) & 0xF);
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        float s = f[0] * xl[m][0];
#pragma unroll
                        for (int t = 1; t < 4; ++t) s = __fmaf_rn(f[t], xl[m][t], s);
#pragma unroll
                        for (int t = 0; t < 4; ++t) s = __fmaf_rn(f[4 + t], xh[m][t], s);
                        acc[m][r] = __fmaf_rn(d, s, acc[m][r]);
                    }
                } else if (FMT == FMT_Q4_K) {
                    const uint8_t* blk = row + pp * 144;
                    const uint32_t hdr = *reinterpret_cast<const uint32_t*>(blk);
                    const uint32_t s0 = *reinterpret_cast<const uint32_t*>(blk + 4);
                    const uint32_t s1 = *reinterpret_cast<const uint32_t*>(blk + 8);
                    const uint32_t s2 = *reinterpret_cast<const uint32_t*>(blk + 12);
                    const uint32_t v = *reinterpret_cast<const uint32_t*>(blk + 16 + lane * 4);
                    int sc0, mn0, sc1, mn1;
                    q4k_pair(s0, s1, s2, q4k_j0, sc0, mn0);
                    q4k_pair(s0, s1, s2, q4k_j0 + 1, sc1, mn1);
                    const float d = __half2float(__ushort_as_half((unsigned short)(hdr & 0xFFFF)));
                    const float dmin = __half2float(__ushort_as_half((unsigned short)(hdr >> 16)));
                    const float ds0 = d * (float)sc0, dm0 = dmin * (float)mn0;
                    const float ds1 = d * (float)sc1, dm1 = dmin * (float)mn1;
                    float f[8];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        f[t] = code_f((v >> (8 * t)) & 0xF);
                        f[4 + t] = code_f((v >> (8 * t + 4)) & 0xF);
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        float sl = f[0] * xl[m][0];
#pragma unroll
                        for (int t = 1; t < 4; ++t) sl = __fmaf_rn(f[t], xl[m][t], sl);
                        float sh = f[4] * xh[m][0];
#pragma unroll
                        for (int t = 1; t < 4; ++t) sh = __fmaf_rn(f[4 + t], xh[m][t], sh);
                        float a = acc[m][r];
                        a = __fmaf_rn(ds0, sl, a);
                        a = __fmaf_rn(-dm0, sxl[m], a);
                        a = __fmaf_rn(ds1, sh, a);
                        a = __fmaf_rn(-dm1, sxh[m], a);
                        acc[m][r] = a;
                    }
                } else {
                    const float* srow =
                        reinterpret_cast<const float*>(stg + p.sb_off + r * p.sb_stride);
                    const float* brow =
                        reinterpret_cast<const float*>(stg + p.sb_off + (R + r) * p.sb_stride);
                    const int g = (pp * kPass + lane * 8) >> p.log2gs;
                    const float sc = srow[g], bi = brow[g];
                    float f[8];
                    if (FMT == FMT_AFF_U8) {
                        const uint2 v = *reinterpret_cast<const uint2*>(row + pp * 256 + lane * 8);
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            f[t] = code_f((v.x >> (8 * t)) & 0xFF);
                            f[4 + t] = code_f((v.y >> (8 * t)) & 0xFF);
                        }
                    } else {
                        const uint32_t v =
                            *reinterpret_cast<const uint32_t*>(row + pp * 128 + lane * 4);
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = code_f((v >> (4 * e)) & 0xF);
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        float s = f[0] * xl[m][0];
#pragma unroll
                        for (int t = 1; t < 4; ++t) s = __fmaf_rn(f[t], xl[m][t], s);
#pragma unroll
                        for (int t = 0; t < 4; ++t) s = __fmaf_rn(f[4 + t], xh[m][t], s);
                        float a = __fmaf_rn(sc, s, acc[m][r]);
                        acc[m][r] = __fmaf_rn(bi, sxl[m] + sxh[m], a);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[st]));

        constexpr int V = MT * R;
        float vals[V];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < R; ++r) vals[m * R + r] = acc[m][r];
        butterfly<V>(vals, lane);
        constexpr int kSpan = 32 / V;
        if ((lane % kSpan) == 0) {
            const int v = lane / kSpan;
            const int m = v / R, r = v % R;
            if (m < p.M && r < rows) {
                const long long o = (long long)m * p.N + row0 + r;
                if (p.KS == 1)
                    p.out[wi][o] = vals[0];
                else
                    p.partial[((long long)(ks * p.nw + wi) * p.M) * p.N + o] = vals[0];
            }
        }
    }
}

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
struct Plan {
    bool fast;
    int MT, R, KS, klen, S, stage_bytes, q_stride, sb_stride, sb_off, smem;
};

int ilog2(int v) {
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

Plan make_plan(const DevCtx& dc, const GemvArgs& a, int Mc) {
    Plan pl{};
    pl.fast = false;
    const bool affine = (a.fmt == FMT_AFF_U8 || a.fmt == FMT_AFF_PACKED);
    pl.MT = Mc <= 1 ? 1 : Mc <= 2 ? 2 : Mc <= 4 ? 4 : 8;
    pl.R = pl.MT <= 2 ? 8 : 4;
    if (a.K % kPass != 0) return pl;
    for (int i = 0; i < a.nw; ++i)
        if (!aligned16(a.w[i])) return pl;
    const long long qrow = (long long)(a.K / kPass) * q_bytes_per_pass(a.fmt);
    if (qrow % 16) return pl;
    if (affine) {
        if (a.gs < 8) return pl;
        const int G = (int)(a.K / a.gs);
        if (G % 4 != 0 || !aligned16(a.scales) || !aligned16(a.biases)) return pl;
    }
    // k-slices: x for MT inputs must fit in kXMaxBytes.
    int KS = 1;
    for (;; ++KS) {
        if (KS > 8) return pl;
        if (a.K % KS) continue;
        const long long klen = a.K / KS;
        if (klen % kPass) continue;
        if (affine && (klen % a.gs || (klen / a.gs) % 4)) continue;
        if ((long long)pl.MT * klen * 4 <= (long long)kXMaxBytes) break;
    }
    pl.KS = KS;
    pl.klen = (int)(a.K / KS);
    pl.q_stride = (pl.klen / kPass) * q_bytes_per_pass(a.fmt);
    pl.sb_stride = affine ? (pl.klen / a.gs) * 4 : 0;
    pl.sb_off = pl.R * pl.q_stride;
    int stage = pl.sb_off + 2 * pl.R * pl.sb_stride + 16;
    pl.stage_bytes = (stage + 127) & ~127;
    const int x_bytes = (pl.MT * pl.klen * 4 + 127) & ~127;
    const int avail = dc.max_smem_optin - x_bytes;
    int S = avail / (pl.stage_bytes + 16);
    S = std::min(S, kMaxStages);
    if (S < 2) return pl;
    pl.S = S;
    pl.smem = x_bytes + S * pl.stage_bytes + 2 * S * 8;
    pl.fast = true;
    return pl;
}

template <int FMT, int MT, int R>
int launch_fast(const DevCtx& dc, const KParams& kp, int grid_x, int smem, cudaStream_t s) {
    auto kern = gemv_kernel<FMT, MT, R>;
    static int configured_dev[64] = {0};  // smem opt-in done per device (+1 tag)
    if (dc.device >= 0 && dc.device < 64 && configured_dev[dc.device] < smem) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dc.max_smem_optin);
        if (e != cudaSuccess) return cuda_fail(e);
        configured_dev[dc.device] = dc.max_smem_optin;
    }
    kern<<<dim3(grid_x, kp.KS), kThreads, smem, s>>>(kp);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

template <int FMT>
int dispatch_fast(const DevCtx& dc, const KParams& kp, const Plan& pl, int grid_x, cudaStream_t s) {
    switch (pl.MT) {
        case 1: return launch_fast<FMT, 1, 8>(dc, kp, grid_x, pl.smem, s);
        case 2: return launch_fast<FMT, 2, 8>(dc, kp, grid_x, pl.smem, s);
        case 4: return launch_fast<FMT, 4, 4>(dc, kp, grid_x, pl.smem, s);
        default: return launch_fast<FMT, 8, 4>(dc, kp, grid_x, pl.smem, s);
    }
}

template <int FMT>
int launch_general(const DevCtx& dc, const KParams& kp, cudaStream_t s) {
    const long long rows = (long long)kp.nw * kp.N;
    const long long blocks = std::min<long long>((rows + 7) / 8, (long long)dc.num_sms * 16);
    gemv_general_kernel<FMT><<<(int)blocks, 256, 0, s>>>(kp);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

KParams base_params(const DevCtx& dc, const GemvArgs& a) {
    KParams kp{};
    kp.w[0] = a.w[0];
    kp.w[1] = a.nw > 1 ? a.w[1] : a.w[0];
    kp.s = a.scales;
    kp.b = a.biases;
    kp.N = (int)a.N;
    kp.K = (int)a.K;
    kp.nw = a.nw;
    kp.log2gs = (a.fmt == FMT_AFF_U8 || a.fmt == FMT_AFF_PACKED) ? ilog2(a.gs) : 0;
    kp.G = (a.fmt == FMT_AFF_U8 || a.fmt == FMT_AFF_PACKED) ? (int)(a.K / a.gs) : 0;
    switch (a.fmt) {
        case FMT_Q4_0: kp.q_row_bytes = a.K / 32 * 18; break;
        case FMT_Q4_K: kp.q_row_bytes = a.K / 256 * 144; break;
        case FMT_AFF_U8: kp.q_row_bytes = a.K; break;
        default: kp.q_row_bytes = a.K / 2; break;
    }
    kp.err = dc.err;
    return kp;
}

}  // namespace

size_t gemv_workspace_bytes(const DevCtx& dc, const GemvArgs& a) {
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
    for (long long m0 = 0; m0 < a.M; m0 += 8) {
        const int Mc = (int)std::min<long long>(8, a.M - m0);
        KParams kp = base_params(dc, a);
        kp.M = Mc;
        kp.x = a.x + m0 * a.K;
        kp.out[0] = a.y[0] + m0 * a.N;
        kp.out[1] = (a.nw > 1 ? a.y[1] : a.y[0]) + m0 * a.N;
        const Plan pl = make_plan(dc, a, Mc);
        int rc;
        if (!pl.fast) {
            switch (a.fmt) {
                case FMT_Q4_0: rc = launch_general<FMT_Q4_0>(dc, kp, s); break;
                case FMT_Q4_K: rc = launch_general<FMT_Q4_K>(dc, kp, s); break;
                case FMT_AFF_U8: rc = launch_general<FMT_AFF_U8>(dc, kp, s); break;
                default: rc = launch_general<FMT_AFF_PACKED>(dc, kp, s); break;
            }
            if (rc != QG_OK) return rc;
            continue;
        }
        kp.KS = pl.KS;
        kp.klen = pl.klen;
        kp.passes = pl.klen / kPass;
        kp.chunks_per_w = (int)((a.N + pl.R - 1) / pl.R);
        kp.total_chunks = kp.chunks_per_w * a.nw;
        kp.S = pl.S;
        kp.stage_bytes = pl.stage_bytes;
        kp.q_stride = pl.q_stride;
        kp.sb_stride = pl.sb_stride;
        kp.sb_off = pl.sb_off;
        if (pl.KS > 1) {
            const size_t need = (size_t)pl.KS * a.nw * Mc * (size_t)a.N * sizeof(float);
            if (!ws || ws_bytes < need) return QG_ERR_WORKSPACE;
            kp.partial = static_cast<float*>(ws);
        }
        const int grid_x = std::max(1, std::min(kp.total_chunks, dc.num_sms / pl.KS));
        switch (a.fmt) {
            case FMT_Q4_0: rc = dispatch_fast<FMT_Q4_0>(dc, kp, pl, grid_x, s); break;
            case FMT_Q4_K: rc = dispatch_fast<FMT_Q4_K>(dc, kp, pl, grid_x, s); break;
            case FMT_AFF_U8: rc = dispatch_fast<FMT_AFF_U8>(dc, kp, pl, grid_x, s); break;
            default: rc = dispatch_fast<FMT_AFF_PACKED>(dc, kp, pl, grid_x, s); break;
        }
        if (rc != QG_OK) return rc;
        if (pl.KS > 1) {
            const long long MN = (long long)Mc * a.N;
            const long long blocks = std::min<long long>((a.nw * MN + 255) / 256, dc.num_sms * 8);
            splitk_finalize<<<(int)blocks, 256, 0, s>>>(kp.partial, kp.out[0], kp.out[1], a.nw,
                                                         pl.KS, MN);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return cuda_fail(e);
        }
    }
    return QG_OK;
}

}  // namespace qg
