// Internal declarations shared by the library's translation units:
// inline-PTX helpers (mbarrier, 1-D TMA bulk copy, timers) and the launchers
// each .cu file exports to the C-ABI layer in qg_api.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "qgemv.h"

namespace qg {

// ---------------------------------------------------------------- error codes
// Codes a kernel writes into the per-device error word (bit mask).
enum : unsigned {
    DEVERR_WAIT_FULL = 1u,      // consumer gave up waiting for a stage to land
    DEVERR_WAIT_EMPTY = 2u,     // producer gave up waiting for a stage to drain
    DEVERR_WAIT_DRAIN = 4u,     // copies still in flight after an error
    DEVERR_SELFTEST = 8u,       // the self-test wait ran out (expected)
    DEVERR_TC_WAIT = 16u,       // a tensor-core pipeline role gave up waiting
};

// Bounded waits give up after this many nanoseconds.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

// ------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete; false after
// `limit_ns` without completion (the caller then records an error).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// As mbar_try_wait, but a thread whose phase is not complete is suspended
// until it completes or about `hint_ns` pass, instead of returning at once:
// waiting warps then take no issue slots from the warps they share a
// scheduler with.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// mbar_wait for waits off the critical path: suspended between polls.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity,
                                                unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 8; ++i)
            if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// L2 policy for data read exactly once (weights): evict first.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D TMA bulk copy global -> shared, completion signalled on `bar` as
// transaction bytes. dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Bulk prefetch of global memory into L2 (no completion to wait for).
// src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void report_error(unsigned* err, unsigned code) {
    if (err) atomicOr(err, code);
}

// ----------------------------------------------------------- launch plumbing
struct DevCtx {
    int device;
    int num_sms;
    int max_smem_optin;   // bytes of dynamic shared memory a block may opt into
    int smem_per_sm;      // shared memory per multiprocessor
    int reserved_smem;    // shared memory the system reserves per block
    unsigned* err;        // device address of this device's error word
};

// Process-wide launch options set through qg_set_option().
long long launch_option(int option);

// ----------------------------------------------------------------- launchers
// GEMV family (gemv.cu). fmt: see GemvFmt. Returns a qg_status.
// FMT_AF4: the prepared AF4-g64 layout (qmm_af4_g64); only the
// register-resident-x kernel reads it through GemvFmt.
enum GemvFmt : int { FMT_Q4_0 = 0, FMT_Q4_K = 1, FMT_AFF_U8 = 2, FMT_AFF_PACKED = 3, FMT_AF4 = 4 };

struct GemvArgs {
    int fmt;
    int nw;                    // 1, or 2 for the fused dual projection
    const uint8_t* w[2];
    float* y[2];
    const float* x;
    const float* scales;       // affine only
    const float* biases;       // affine only
    int64_t M, N, K;
    int gs;                    // affine only
    // x is written by the kernel launched just before on the stream: the
    // register-resident-x kernel is then launched as its programmatic
    // dependent and waits for it before reading x, whatever QG_OPT_PDL says.
    bool x_from_prev;
    // The call runs alone: the caller waits for it before anything else is
    // queued. The register-resident-x kernel then gives its CTA all of the
    // SM's shared memory (no room is kept for the next call's CTAs) and never
    // takes the four-warp shape meant for overlapping calls.
    bool isolated;
};

size_t gemv_workspace_bytes(const DevCtx& dc, const GemvArgs& a);
int gemv_launch(const DevCtx& dc, const GemvArgs& a, void* ws, size_t ws_bytes, cudaStream_t s);
bool gemv_xreg_only(const DevCtx& dc, const GemvArgs& a);

// dst[0..n) = src[0..n) (f32) by a kernel; src is mapped host memory, n a
// multiple of 4, both pointers 16-byte aligned (host_io.cu).
int fetch_host_launch(const DevCtx& dc, const float* src, float* dst, long long n,
                      cudaStream_t s);

// The prepared AF4-g64 layout: repack from codes and bf16 scale / bias bits
// (af4.cu), and the qmm that reads it, M <= 32 (af4_gemv.cu).
int af4_prepare_launch(const DevCtx& dc, const uint8_t* codes, const uint16_t* sb,
                       const uint16_t* bb, uint32_t* plane, uint32_t* meta, long long N,
                       long long K, cudaStream_t s);
int af4_gemv_launch(const DevCtx& dc, const float* x, const uint32_t* plane, const uint32_t* meta,
                    float* y, long long M, long long N, long long K, cudaStream_t s);
// qmm_af4_g64 on the register-resident-x kernel for M <= 2 (gemv_xreg_af4.cu);
// QG_ERR_UNSUPPORTED, with nothing enqueued, when the shape or alignment does
// not suit it.
int af4_xreg_launch(const DevCtx& dc, const float* x, const uint32_t* plane, const uint32_t* meta,
                    float* y, long long M, long long N, long long K, cudaStream_t s);

// Affine prefill on the tensor cores (prefill.cu). Eligibility depends on the
// shape, the group size, the code and activation pointers' alignment and the
// QG_OPT_PREFILL_MIN_M option.
bool prefill_eligible(const DevCtx& dc, const GemvArgs& a);
size_t prefill_workspace_bytes(const GemvArgs& a);
int prefill_launch(const DevCtx& dc, const GemvArgs& a, void* ws, size_t ws_bytes, cudaStream_t s);

// Q4_0 / Q4_K prefill (prefill_repack.cu): the weights rewritten as packed
// affine codes with group size 32 in the workspace, then the affine prefill.
bool quant_prefill_eligible(const DevCtx& dc, const GemvArgs& a);
size_t quant_prefill_workspace_bytes(const GemvArgs& a);
int quant_prefill_launch(const DevCtx& dc, const GemvArgs& a, void* ws, size_t ws_bytes,
                         cudaStream_t s);

// Copies and dequantization (elementwise.cu).
int qkv_split_launch(const DevCtx& dc, const float* qkv, float* q, float* k, float* v,
                     int64_t seq, int64_t q_sp, int64_t k_sp, int64_t v_sp, cudaStream_t s);
int dequant_launch(const DevCtx& dc, int fmt, const uint8_t* w, const float* scales,
                   const float* biases, float* out, int64_t N, int64_t K, int gs,
                   cudaStream_t s);
int selftest_wait_launch(const DevCtx& dc, long long timeout_ns, cudaStream_t s);

// qgemv_q4_k restricted to its CUDA-core kernels (never the tensor-core
// prefill, whatever M and the workspace): same validation, same status codes.
int q4_k_cuda_core(const void* w, const float* x, float* y, int64_t M, int64_t N, int64_t K,
                   void* ws, size_t ws_bytes, qg_stream_t stream);

// Workspace of the CUDA-core path alone (qg_workspace_size also covers the
// Q4_0 / Q4_K tensor-core prefill, which calls with a smaller workspace skip).
int cuda_core_workspace_size(int op, int64_t M, int64_t N, int64_t K, size_t* bytes);

// Record a CUDA error for qg_last_cuda_error() and return QG_ERR_CUDA.
int cuda_fail(cudaError_t e);

}  // namespace qg
