// Bandwidth kernels: the fused-QKV split (a pure bit copy) and the
// dequantization exports (bit-exact f32 weights).
//
// Pages: qkv_split.rs (mlx-native 0.7.1) for the split - per token the fused
// row is [Q | K | V] and every element is written to exactly one output;
// qmm_affine.rs (mlx-native 0.21.1) for dequantize-then-matmul as a
// composition check; the Q4_0 / Q4_K block layouts of fused_dual_proj_q4_0.rs
// and q4_k_gemv_v2.rs.
#include <cuda_fp16.h>

#include <algorithm>

#include "qg_internal.cuh"

namespace qg {
namespace {

// One block per row (grid-strided over rows); 16-byte vectors when every span
// and pointer allows it, else 32-bit words. Loads of a batch are issued
// before its stores so that several 16-byte requests per thread are in flight.
template <typename T>
__global__ void __launch_bounds__(256) qkv_split_kernel(const T* __restrict__ src, T* __restrict__ q,
                                                         T* __restrict__ k, T* __restrict__ v,
                                                         long long seq, long long q_sp,
                                                         long long k_sp, long long v_sp) {
    constexpr int kUnroll = 4;
    const long long ch = q_sp + k_sp + v_sp;
    const long long qk = q_sp + k_sp;
    for (long long t = blockIdx.x; t < seq; t += gridDim.x) {
        const T* row = src + t * ch;
        for (long long j0 = threadIdx.x; j0 < ch; j0 += (long long)blockDim.x * kUnroll) {
            T val[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const long long j = j0 + (long long)u * blockDim.x;
                if (j < ch) val[u] = __ldcs(row + j);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const long long j = j0 + (long long)u * blockDim.x;
                if (j >= ch) break;
                T* dst = (j < q_sp) ? q + t * q_sp + j
                         : (j < qk) ? k + t * k_sp + (j - q_sp)
                                    : v + t * v_sp + (j - qk);
                __stcs(dst, val[u]);
            }
        }
    }
}

__device__ __forceinline__ float half_bits_to_float(unsigned lo, unsigned hi) {
    return __half2float(__ushort_as_half((unsigned short)(lo | (hi << 8))));
}

// One thread per Q4_0 block: 32 outputs w = (q - 8) * d (an exact product).
__global__ void dequant_q4_0_kernel(const uint8_t* __restrict__ w, float* __restrict__ out,
                                    long long nblocks) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nblocks;
         i += (long long)gridDim.x * blockDim.x) {
        const uint8_t* blk = w + i * 18;
        const float d = half_bits_to_float(blk[0], blk[1]);
        float* o = out + i * 32;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const uint8_t byte = blk[2 + j];
            o[j] = __fmul_rn((float)((int)(byte & 15) - 8), d);
            o[16 + j] = __fmul_rn((float)((int)(byte >> 4) - 8), d);
        }
    }
}

// One thread per (super-block, nibble chunk c): sub-blocks 2c and 2c+1.
// w = (d*sc)*q - dmin*m; both products are exact, so the fma rounds once.
__global__ void dequant_q4_k_kernel(const uint8_t* __restrict__ w, float* __restrict__ out,
                                    long long nsuper) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nsuper * 4;
         i += (long long)gridDim.x * blockDim.x) {
        const long long sb = i >> 2;
        const int c = (int)(i & 3);
        const uint8_t* blk = w + sb * 144;
        const float d = half_bits_to_float(blk[0], blk[1]);
        const float dmin = half_bits_to_float(blk[2], blk[3]);
        const uint8_t* s12 = blk + 4;
        float ds[2], dm[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = 2 * c + h;
            int sc, mn;
            if (j < 4) {
                sc = s12[j] & 63;
                mn = s12[j + 4] & 63;
            } else {
                sc = (s12[j + 4] & 15) | ((s12[j - 4] >> 6) << 4);
                mn = (s12[j + 4] >> 4) | ((s12[j] >> 6) << 4);
            }
            ds[h] = __fmul_rn(d, (float)sc);
            dm[h] = __fmul_rn(dmin, (float)mn);
        }
        const uint8_t* qs = blk + 16 + 32 * c;
        float* o = out + sb * 256 + 64 * c;
#pragma unroll 8
        for (int l = 0; l < 32; ++l) {
            const uint8_t byte = qs[l];
            o[l] = __fmaf_rn(ds[0], (float)(byte & 15), -dm[0]);
            o[32 + l] = __fmaf_rn(ds[1], (float)(byte >> 4), -dm[1]);
        }
    }
}

// One thread per output element: w = fma(q, s, b), one rounding.
__global__ void dequant_affine_kernel(const uint8_t* __restrict__ q, const float* __restrict__ s,
                                      const float* __restrict__ b, float* __restrict__ out,
                                      long long N, long long K, int log2gs, int packed) {
    const long long total = N * K;
    const long long G = K >> log2gs;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long n = i / K, kk = i - n * K;
        int code;
        if (packed) {
            const uint8_t byte = q[n * (K >> 1) + (kk >> 1)];
            code = (kk & 1) ? (byte >> 4) : (byte & 15);
        } else {
            code = q[i];
        }
        const long long g = n * G + (kk >> log2gs);
        out[i] = __fmaf_rn((float)code, s[g], b[g]);
    }
}

__global__ void selftest_wait_kernel(unsigned* err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        fence_mbar_init();
        // Nobody ever arrives: the bounded wait must give up and report.
        if (!mbar_wait(smem_addr(&bar), 0, limit_ns)) report_error(err, DEVERR_SELFTEST);
    }
}

int grid_for(const DevCtx& dc, long long work, int per_block) {
    const long long need = (work + per_block - 1) / per_block;
    return (int)std::max<long long>(1, std::min<long long>(need, (long long)dc.num_sms * 16));
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

int qkv_split_launch(const DevCtx& dc, const float* qkv, float* q, float* k, float* v,
                     int64_t seq, int64_t q_sp, int64_t k_sp, int64_t v_sp, cudaStream_t s) {
    const int blocks = (int)std::max<long long>(1, std::min<long long>(seq, (long long)dc.num_sms * 8));
    const bool vec = (q_sp % 4 == 0) && (k_sp % 4 == 0) && (v_sp % 4 == 0) && al16(qkv) && al16(q) &&
                     al16(k) && al16(v);
    if (vec) {
        qkv_split_kernel<uint4><<<blocks, 256, 0, s>>>(
            reinterpret_cast<const uint4*>(qkv), reinterpret_cast<uint4*>(q),
            reinterpret_cast<uint4*>(k), reinterpret_cast<uint4*>(v), seq, q_sp / 4, k_sp / 4,
            v_sp / 4);
    } else {
        qkv_split_kernel<unsigned><<<blocks, 256, 0, s>>>(
            reinterpret_cast<const unsigned*>(qkv), reinterpret_cast<unsigned*>(q),
            reinterpret_cast<unsigned*>(k), reinterpret_cast<unsigned*>(v), seq, q_sp, k_sp, v_sp);
    }
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

int dequant_launch(const DevCtx& dc, int fmt, const uint8_t* w, const float* scales,
                   const float* biases, float* out, int64_t N, int64_t K, int gs,
                   cudaStream_t s) {
    if (fmt == FMT_Q4_0) {
        const long long nb = N * (K / 32);
        dequant_q4_0_kernel<<<grid_for(dc, nb, 256), 256, 0, s>>>(w, out, nb);
    } else if (fmt == FMT_Q4_K) {
        const long long ns = N * (K / 256);
        dequant_q4_k_kernel<<<grid_for(dc, ns * 4, 256), 256, 0, s>>>(w, out, ns);
    } else {
        int l2 = 0;
        while ((1 << l2) < gs) ++l2;
        dequant_affine_kernel<<<grid_for(dc, N * K, 256), 256, 0, s>>>(
            w, scales, biases, out, N, K, l2, fmt == FMT_AFF_PACKED ? 1 : 0);
    }
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

int selftest_wait_launch(const DevCtx& dc, long long timeout_ns, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(dc.err, (unsigned long long)timeout_ns);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

}  // namespace qg
