// Q4_0 and Q4_K matmul for many activation rows (prefill) on the tensor
// cores, through the affine prefill kernel of prefill.cu.
//
// Pages: fused_dual_proj_q4_0.rs (mlx-native 0.9.1) and q4_k_gemv_v2.rs
// (ferrum-kernels 0.7.7) define the formats; their GEMVs take one activation
// row. Both formats are affine per 32 weights:
//
//     Q4_0 block b:       w = d * q - 8 d                 (q = 0..15)
//     Q4_K sub-block j:   w = (d * sc_j) * q - dmin * m_j
//
// so a weight matrix is an affine-quantized one with group size 32, scale
// s = d (or d * sc_j) and bias b = -8 d (or -dmin * m_j), every product exact
// in f32. repack_kernel writes that form, codes packed two per byte (low
// nibble = even k) with f32 scales and biases [N][K/32], into the caller's
// workspace; the affine prefill kernel then computes y with exact integer
// codes on the tensor cores and scale and bias in its f32 epilogue, within
// the prefill tolerance 2e-3 * sum_k |x_k w_k| + 1e-6.
#include <cuda_fp16.h>

#include <algorithm>

#include "qg_internal.cuh"

namespace qg {
namespace {

constexpr int kRepackThreads = 256;

__device__ __forceinline__ float half_bits(unsigned lo, unsigned hi) {
    return __half2float(__ushort_as_half((unsigned short)(lo | (hi << 8))));
}

// One thread per (row n, 32-weight group g): 16 packed code bytes, s, b.
template <int FMT>
__global__ void __launch_bounds__(kRepackThreads) repack_kernel(const uint8_t* __restrict__ w,
                                                                uint8_t* __restrict__ codes,
                                                                float* __restrict__ sc,
                                                                float* __restrict__ bi, int N,
                                                                int K) {
    const int G = K >> 5;
    const long long total = (long long)N * G;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const int n = (int)(t / G), g = (int)(t - (long long)n * G);
        uint8_t q[32];
        float s, b;
        if (FMT == FMT_Q4_0) {
            const uint8_t* blk = w + (long long)n * G * 18 + (long long)g * 18;
            const float d = half_bits(blk[0], blk[1]);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                q[i] = blk[2 + i] & 15;
                q[16 + i] = blk[2 + i] >> 4;
            }
            s = d;
            b = -8.0f * d;  // exact: a power-of-two multiple
        } else {
            const int sb = g >> 3, j = g & 7;  // super-block, sub-block
            const uint8_t* blk = w + (long long)n * (K / 256) * 144 + (long long)sb * 144;
            const float d = half_bits(blk[0], blk[1]);
            const float dmin = half_bits(blk[2], blk[3]);
            const uint8_t* s12 = blk + 4;
            int scv, mnv;
            if (j < 4) {
                scv = s12[j] & 63;
                mnv = s12[j + 4] & 63;
            } else {
                scv = (s12[j + 4] & 15) | ((s12[j - 4] >> 6) << 4);
                mnv = (s12[j + 4] >> 4) | ((s12[j] >> 6) << 4);
            }
            const uint8_t* qs = blk + 16 + 32 * (j >> 1);
            const int sh = 4 * (j & 1);  // even sub-block: low nibbles, odd: high
#pragma unroll
            for (int i = 0; i < 32; ++i) q[i] = (qs[i] >> sh) & 15;
            s = d * (float)scv;      // exact: 11-bit by 6-bit product
            b = -(dmin * (float)mnv);
        }
        uint4 out;
        uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t v = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int e = 8 * k + 2 * i;
                v |= (uint32_t)(q[e] | (q[e + 1] << 4)) << (8 * i);
            }
            o[k] = v;
        }
        *reinterpret_cast<uint4*>(codes + (long long)n * (K / 2) + (long long)g * 16) = out;
        sc[t] = s;
        bi[t] = b;
    }
}

struct RepackLayout {
    size_t codes, sc, bi, total;
};

RepackLayout repack_layout(long long N, long long K) {
    auto up = [](size_t v) { return (v + 1023) & ~(size_t)1023; };
    RepackLayout L{};
    L.codes = 0;
    L.sc = up((size_t)N * K / 2);
    L.bi = L.sc + up((size_t)N * (K / 32) * 4);
    L.total = L.bi + up((size_t)N * (K / 32) * 4);
    return L;
}

// The affine problem the repacked matrix poses (pointers filled by the caller).
GemvArgs affine_args(const GemvArgs& a) {
    GemvArgs b{};
    b.fmt = FMT_AFF_PACKED;
    b.nw = 1;
    b.x = a.x;
    b.M = a.M;
    b.N = a.N;
    b.K = a.K;
    b.gs = 32;
    return b;
}

}  // namespace

bool quant_prefill_eligible(const DevCtx& dc, const GemvArgs& a) {
    if (a.fmt != FMT_Q4_0 && a.fmt != FMT_Q4_K) return false;
    if (a.K % 32) return false;
    GemvArgs b = affine_args(a);
    // Stand-in 16-byte aligned code/scale pointers: the workspace provides them.
    static const uint8_t probe[16] __attribute__((aligned(16))) = {0};
    b.w[0] = probe;
    b.scales = b.biases = reinterpret_cast<const float*>(probe);
    return prefill_eligible(dc, b);
}

size_t quant_prefill_workspace_bytes(const GemvArgs& a) {
    return repack_layout(a.N, a.K).total + prefill_workspace_bytes(affine_args(a));
}

int quant_prefill_launch(const DevCtx& dc, const GemvArgs& a, void* ws, size_t ws_bytes,
                         cudaStream_t s) {
    const RepackLayout L = repack_layout(a.N, a.K);
    if (!ws || ws_bytes < quant_prefill_workspace_bytes(a)) return QG_ERR_WORKSPACE;
    uint8_t* base = static_cast<uint8_t*>(ws);
    uint8_t* codes = base + L.codes;
    float* sc = reinterpret_cast<float*>(base + L.sc);
    float* bi = reinterpret_cast<float*>(base + L.bi);
    const long long total = a.N * (a.K / 32);
    const int blocks = (int)std::min<long long>((total + kRepackThreads - 1) / kRepackThreads,
                                                (long long)dc.num_sms * 16);
    // One matrix at a time through the same workspace (stream order keeps the
    // second repack behind the first matrix's prefill).
    for (int i = 0; i < a.nw; ++i) {
        if (a.fmt == FMT_Q4_0)
            repack_kernel<FMT_Q4_0><<<blocks, kRepackThreads, 0, s>>>(a.w[i], codes, sc, bi,
                                                                       (int)a.N, (int)a.K);
        else
            repack_kernel<FMT_Q4_K><<<blocks, kRepackThreads, 0, s>>>(a.w[i], codes, sc, bi,
                                                                       (int)a.N, (int)a.K);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e);
        GemvArgs b = affine_args(a);
        b.w[0] = codes;
        b.scales = sc;
        b.biases = bi;
        b.y[0] = a.y[i];
        const int rc = prefill_launch(dc, b, base + L.total, ws_bytes - L.total, s);
        if (rc != QG_OK) return rc;
    }
    return QG_OK;
}

}  // namespace qg
