// The prepared 4-bit affine layout with groups of 64 ("AF4-g64"): the repack
// tool that writes it (this file) and the qmm that reads it (af4_gemv.cu).
//
// Page: qmm_affine.rs (mlx-native 0.21.1): prepare_af4_g64 in the test module
// defines the layout, dispatch_qmm_affine_t_packed_simd4_b4_gs64_bf16 the
// call (M <= 32, N % 64 == 0, K % 64 == 0, u32 weights and metadata).
//  - plane u32 [N/64][K/32][64][4]: word c of (row r, 32-group g) holds, for
//    pair p = 0..3 and e0 = 16 (p >> 1) + 4c + 2 (p & 1), code e0 of the
//    group in bits 4p.. and code e0 + 1 in bits 16 + 4p..;
//  - metadata u32 [N/64][K/64][64]: bf16 scale | bf16 bias << 16.
#include <algorithm>

#include "qg_internal.cuh"

namespace qg {
namespace {

constexpr int kThreads = 256;

// One thread per (row, 32-group, word).
__global__ void __launch_bounds__(kThreads) prepare_plane_kernel(const uint8_t* __restrict__ codes,
                                                                  uint32_t* __restrict__ plane,
                                                                  int N, int K) {
    const int G32 = K / 32;
    const long long total = (long long)N * G32 * 4;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(t & 3);
        const long long rg = t >> 2;
        const int row = (int)(rg / G32), g = (int)(rg - (long long)row * G32);
        const uint8_t* src = codes + (long long)row * K + g * 32;
        uint32_t word = 0;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int e0 = 16 * (p >> 1) + 4 * c + 2 * (p & 1);
            word |= (uint32_t)(src[e0] & 15) << (4 * p);
            word |= (uint32_t)(src[e0 + 1] & 15) << (16 + 4 * p);
        }
        plane[(((long long)(row / 64) * G32 + g) * 64 + row % 64) * 4 + c] = word;
    }
}

// One thread per (row, 64-group).
__global__ void __launch_bounds__(kThreads) prepare_meta_kernel(const uint16_t* __restrict__ sb,
                                                                 const uint16_t* __restrict__ bb,
                                                                 uint32_t* __restrict__ meta, int N,
                                                                 int K) {
    const int G64 = K / 64;
    const long long total = (long long)N * G64;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const int row = (int)(t / G64), g = (int)(t - (long long)row * G64);
        meta[((long long)(row / 64) * G64 + g) * 64 + row % 64] =
            (uint32_t)sb[t] | ((uint32_t)bb[t] << 16);
    }
}

unsigned blocks_for(const DevCtx& dc, long long total) {
    return (unsigned)std::max<long long>(
        1, std::min<long long>((total + kThreads - 1) / kThreads, (long long)dc.num_sms * 16));
}

}  // namespace

int af4_prepare_launch(const DevCtx& dc, const uint8_t* codes, const uint16_t* sb,
                       const uint16_t* bb, uint32_t* plane, uint32_t* meta, long long N,
                       long long K, cudaStream_t s) {
    prepare_plane_kernel<<<blocks_for(dc, N * (K / 32) * 4), kThreads, 0, s>>>(codes, plane, (int)N,
                                                                              (int)K);
    prepare_meta_kernel<<<blocks_for(dc, N * (K / 64)), kThreads, 0, s>>>(sb, bb, meta, (int)N,
                                                                         (int)K);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

}  // namespace qg
