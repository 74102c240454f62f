// qgemv_q4_k_noalloc: the Q4_K GEMV for callers that cannot allocate device
// memory (for example code running inside a CUDA graph that was captured by
// someone else, a plugin inside a host application that owns every device
// allocation, or a runtime that forbids cudaMalloc after start-up). The
// regular qgemv_q4_k needs a caller-provided workspace for its split-K
// partial sums whenever x for all M rows does not fit in shared memory; this
// variant uses a fixed-size scratch array that lives in the library's own
// device memory instead.
#include <cuda_runtime.h>

#include <mutex>

#include "qg_internal.cuh"

namespace qg {
namespace {

// Largest split-K scratch the entry point can use. Every GPU that loads the
// library holds this array (4 MiB) until the process exits.
constexpr size_t kNoAllocScratchBytes = 4u << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_lock;
void* g_addr[kMaxDev];  // non-null once the lookup has succeeded on that device

// Device address of the scratch array on the current device. The host-side
// name g_noalloc_scratch is only a stand-in for the symbol; the address a
// kernel may use comes from cudaGetSymbolAddress, taken with that device
// current. Only a successful lookup is kept: a failed one (for example a
// first call made inside a stream capture) is retried by the next call.
int scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDev) return QG_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_lock);
    if (!g_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e);
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return QG_OK;
}

}  // namespace
}  // namespace qg

extern "C" int qgemv_q4_k_noalloc(const void* w, const float* x, float* y, int64_t M, int64_t N,
                                  int64_t K, qg_stream_t stream) {
    size_t need = 0;
    int rc = qg::cuda_core_workspace_size(QG_OP_Q4_K, M, N, K, &need);
    if (rc != QG_OK) return rc;
    if (need > qg::kNoAllocScratchBytes) return QG_ERR_WORKSPACE;
    void* scratch = nullptr;
    rc = qg::scratch_address(&scratch);
    if (rc != QG_OK) return rc;
    // The split-K partial sums are fully written before they are read, so
    // nothing in the scratch array needs clearing between calls. The call
    // stays on the CUDA-core kernels for every M: the tensor-core prefill
    // would need scratch for rewritten weights, and has a looser error bound.
    return qg::q4_k_cuda_core(w, x, y, M, N, K, scratch, qg::kNoAllocScratchBytes, stream);
}
