// Moving a call's input from host memory into the device workspace with a
// kernel of this library instead of the copy engine: qgemv_dual_q4_0_host's
// zero-copy route (the host round trip that qkv_split.rs's module doc names
// as the cost to cut). The GEMV that follows is launched as this kernel's
// programmatic dependent: it streams its weights while x is still on its
// way and reads x only after this grid has completed.
#include <algorithm>

#include "qg_internal.cuh"

namespace qg {
namespace {

constexpr int kFetchThreads = 256;

// dst[i] = src[i] for n16 16-byte vectors; src is page-locked host memory
// mapped for the device. Each thread issues all of its loads before its
// stores, so that many requests cross the host link at once.
__global__ void __launch_bounds__(kFetchThreads) fetch_kernel(const float4* __restrict__ src,
                                                               float4* __restrict__ dst,
                                                               long long n16) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int kUnroll = 4;
    const long long stride = (long long)gridDim.x * kFetchThreads;
    for (long long i0 = blockIdx.x * (long long)kFetchThreads + threadIdx.x; i0 < n16;
         i0 += stride * kUnroll) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long i = i0 + u * stride;
            if (i < n16) v[u] = src[i];
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long i = i0 + u * stride;
            if (i < n16) dst[i] = v[u];
        }
    }
}

}  // namespace

int fetch_host_launch(const DevCtx& dc, const float* src, float* dst, long long n,
                      cudaStream_t s) {
    if (n <= 0) return QG_OK;
    if (n % 4 || (reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) % 16)
        return QG_ERR_MISALIGNED;
    // All of the SM's on-chip memory to shared memory, as the GEMV that
    // follows wants it: the GEMV's CTAs may then start beside this kernel's
    // on the same SMs instead of waiting for them to end.
    static int configured[64] = {0};
    if (dc.device >= 0 && dc.device < 64 && !configured[dc.device]) {
        const cudaError_t e = cudaFuncSetAttribute(
            fetch_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return cuda_fail(e);
        configured[dc.device] = 1;
    }
    const long long n16 = n / 4;
    // One vector per thread while that fills at most four CTAs per SM.
    const long long want = (n16 + kFetchThreads - 1) / kFetchThreads;
    const int grid = (int)std::min<long long>(want, 4ll * dc.num_sms);
    fetch_kernel<<<grid, kFetchThreads, 0, s>>>(reinterpret_cast<const float4*>(src),
                                                 reinterpret_cast<float4*>(dst), n16);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

}  // namespace qg
