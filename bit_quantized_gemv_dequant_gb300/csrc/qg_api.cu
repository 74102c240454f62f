// C-ABI entry points declared in include/qgemv.h: argument validation (every
// check happens before anything is enqueued, mirroring the InvalidArgument-
// before-encode contract of the pages' dispatch functions), per-device
// context, and dispatch to the kernels of gemv.cu and elementwise.cu.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "qg_internal.cuh"

namespace qg {

// Per-device error word written by kernels that give up on a bounded wait.
__device__ unsigned g_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;
DevCtx g_ctx[kMaxDevices];
std::once_flag g_once[kMaxDevices];
int g_ctx_rc[kMaxDevices];
thread_local int t_last_cuda_error = 0;
std::atomic<long long> g_opt_pdl{0};
std::atomic<long long> g_opt_prefill_min_m{64};
std::atomic<long long> g_opt_stream{1};
std::atomic<long long> g_opt_stream_warps{0};
std::atomic<long long> g_opt_stream_slots{0};
std::atomic<long long> g_opt_ahead{2};
std::atomic<long long> g_opt_staged_warps{0};
std::atomic<long long> g_opt_prefill_fold{0};
std::atomic<long long> g_opt_xreg{1};
std::atomic<long long> g_opt_xreg_ahead{0};
std::atomic<long long> g_opt_xreg_warps{0};
std::atomic<long long> g_opt_xreg_ctas{0};

int init_ctx(int dev) {
    DevCtx& c = g_ctx[dev];
    c.device = dev;
    cudaError_t e = cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaDeviceGetAttribute(&c.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaDeviceGetAttribute(&c.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaDeviceGetAttribute(&c.reserved_smem, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) return cuda_fail(e);
    c.err = static_cast<unsigned*>(p);
    return QG_OK;
}

// Context of the current device, created on first use.
int current_ctx(const DevCtx** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return QG_ERR_UNSUPPORTED;
    std::call_once(g_once[dev], [dev] { g_ctx_rc[dev] = init_ctx(dev); });
    if (g_ctx_rc[dev] != QG_OK) return g_ctx_rc[dev];
    *out = &g_ctx[dev];
    return QG_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// [a, a+na) and [b, b+nb) (bytes) overlap?
bool overlap(const void* a, long long na, const void* b, long long nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + (uintptr_t)nb && y < x + (uintptr_t)na;
}

constexpr long long kMaxDim = 0x7FFFFFFFLL;

int check_dims(long long M, long long N, long long K) {
    if (M <= 0 || N <= 0 || K <= 0) return QG_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return QG_ERR_UNSUPPORTED;
    return QG_OK;
}

long long weight_bytes(int fmt, long long N, long long K) {
    switch (fmt) {
        case FMT_Q4_0: return N * (K / 32) * 18;
        case FMT_Q4_K: return N * (K / 256) * 144;
        case FMT_AFF_U8: return N * K;
        default: return N * (K / 2);
    }
}

// Shared validation of a GEMV request. Fills nothing; returns a status.
int validate_gemv(const GemvArgs& a) {
    int rc = check_dims(a.M, a.N, a.K);
    if (rc) return rc;
    if (!a.x) return QG_ERR_INVALID_ARG;
    for (int i = 0; i < a.nw; ++i)
        if (!a.w[i] || !a.y[i]) return QG_ERR_INVALID_ARG;
    switch (a.fmt) {
        case FMT_Q4_0:
            if (a.K % 32) return QG_ERR_INVALID_ARG;
            break;
        case FMT_Q4_K:
            if (a.K % 256) return QG_ERR_INVALID_ARG;
            break;
        default:
            if (!a.scales || !a.biases) return QG_ERR_INVALID_ARG;
            if (a.gs < 2 || a.gs > 1024 || (a.gs & (a.gs - 1))) return QG_ERR_INVALID_ARG;
            if (a.K % a.gs) return QG_ERR_INVALID_ARG;
            if (a.fmt == FMT_AFF_PACKED && (a.K & 1)) return QG_ERR_INVALID_ARG;
            if (!aligned(a.scales, 4) || !aligned(a.biases, 4)) return QG_ERR_MISALIGNED;
            break;
    }
    if (!aligned(a.x, 4)) return QG_ERR_MISALIGNED;
    for (int i = 0; i < a.nw; ++i)
        if (!aligned(a.y[i], 4)) return QG_ERR_MISALIGNED;
    // Outputs must not overlap each other or any input.
    const long long xb = a.M * a.K * 4, yb = a.M * a.N * 4, wb = weight_bytes(a.fmt, a.N, a.K);
    for (int i = 0; i < a.nw; ++i) {
        if (overlap(a.y[i], yb, a.x, xb)) return QG_ERR_INVALID_ARG;
        for (int j = 0; j < a.nw; ++j)
            if (overlap(a.y[i], yb, a.w[j], wb)) return QG_ERR_INVALID_ARG;
        if (a.scales) {
            const long long sb = a.N * (a.K / a.gs) * 4;
            if (overlap(a.y[i], yb, a.scales, sb) || overlap(a.y[i], yb, a.biases, sb))
                return QG_ERR_INVALID_ARG;
        }
    }
    if (a.nw == 2 && overlap(a.y[0], yb, a.y[1], yb)) return QG_ERR_INVALID_ARG;
    return QG_OK;
}

int run_gemv(const GemvArgs& a, void* ws, size_t ws_bytes, qg_stream_t stream) {
    int rc = validate_gemv(a);
    if (rc) return rc;
    if (ws && !aligned(ws, 16)) return QG_ERR_MISALIGNED;
    const DevCtx* dc = nullptr;
    rc = current_ctx(&dc);
    if (rc) return rc;
    if (prefill_eligible(*dc, a)) {
        if (prefill_workspace_bytes(a) > (ws ? ws_bytes : 0)) return QG_ERR_WORKSPACE;
        return prefill_launch(*dc, a, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
    }
    // Q4_0 / Q4_K prefill on the tensor cores when the workspace holds the
    // repacked weights; otherwise the CUDA-core path (smaller workspace).
    if (quant_prefill_eligible(*dc, a) && ws && ws_bytes >= quant_prefill_workspace_bytes(a))
        return quant_prefill_launch(*dc, a, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
    if (gemv_workspace_bytes(*dc, a) > (ws ? ws_bytes : 0)) return QG_ERR_WORKSPACE;
    return gemv_launch(*dc, a, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

// Host-buffer calls stage x and the outputs in the workspace after the
// call's own part: [call workspace | x | y_a | y_b], each part starting on a
// 256-byte boundary (relative to the workspace's start).
size_t round256(size_t v) { return (v + 255) & ~(size_t)255; }
size_t host_stage_offset(size_t call_bytes) { return round256(call_bytes); }
size_t host_stage_bytes(const GemvArgs& a) {
    return round256((size_t)(a.M * a.K) * 4) + (size_t)a.nw * round256((size_t)(a.M * a.N) * 4);
}

// Device address of p when it is page-locked host memory mapped for the
// current device; nullptr otherwise (pageable or device memory).
template <class T>
T* mapped_host(T* p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || !at.devicePointer || !at.hostPointer) return nullptr;
    const ptrdiff_t off = reinterpret_cast<const char*>(p) - static_cast<const char*>(at.hostPointer);
    return reinterpret_cast<T*>(static_cast<char*>(at.devicePointer) + off);
}

// A GEMV whose x and outputs are host buffers: returns once the outputs hold
// the result. Zero-copy route when every buffer is mapped page-locked memory
// and every slice runs on the register-resident-x kernel: x is fetched into
// the workspace by a kernel (fetch_host_launch), the GEMV follows as its
// programmatic dependent and stores its outputs straight into host memory.
// Otherwise one cudaMemcpyAsync per buffer through the workspace around an
// ordinary call.
int run_gemv_host(const GemvArgs& a, void* ws, size_t ws_bytes, qg_stream_t stream) {
    int rc = validate_gemv(a);
    if (rc) return rc;
    if (ws && !aligned(ws, 16)) return QG_ERR_MISALIGNED;
    const DevCtx* dc = nullptr;
    rc = current_ctx(&dc);
    if (rc) return rc;
    const size_t stage = host_stage_bytes(a);
    if (!ws || ws_bytes < stage) return QG_ERR_WORKSPACE;
    // The staging area sits at the end of the workspace; the call keeps the
    // part before it.
    const size_t off = (ws_bytes - stage) & ~(size_t)255;
    uint8_t* base = static_cast<uint8_t*>(ws);
    float* xs = reinterpret_cast<float*>(base + off);
    float* ys[2];
    ys[0] = reinterpret_cast<float*>(base + off + round256((size_t)(a.M * a.K) * 4));
    ys[1] = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ys[0]) +
                                     round256((size_t)(a.M * a.N) * 4));
    void* call_ws = off ? ws : nullptr;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t xb = (size_t)(a.M * a.K) * 4, yb = (size_t)(a.M * a.N) * 4;

    GemvArgs d = a;
    d.x = xs;
    d.isolated = true;  // the call is waited for before it returns
    float* ym[2] = {nullptr, nullptr};
    bool direct = mapped_host(a.x) != nullptr && aligned(a.x, 16);
    for (int i = 0; i < a.nw && direct; ++i) {
        ym[i] = mapped_host(a.y[i]);
        direct = ym[i] != nullptr;
    }
    if (direct) {
        GemvArgs t = d;
        t.y[0] = ym[0];
        t.y[1] = ym[1];
        direct = !prefill_eligible(*dc, t) &&
                 !(quant_prefill_eligible(*dc, t) && off >= quant_prefill_workspace_bytes(t)) &&
                 gemv_xreg_only(*dc, t);
        if (direct) d = t;
    }
    if (direct) {
        rc = fetch_host_launch(*dc, mapped_host(a.x), xs, a.M * a.K, s);
        if (rc) return rc;
        d.x_from_prev = true;
        rc = gemv_launch(*dc, d, nullptr, 0, s);
        if (rc) return rc;
    } else {
        d.y[0] = ys[0];
        d.y[1] = ys[1];
        // The call's own workspace need, checked before anything is enqueued
        // (run_gemv's rule: the tensor-core prefill when its workspace fits,
        // else the CUDA-core kernels).
        size_t need = gemv_workspace_bytes(*dc, d);
        if (prefill_eligible(*dc, d))
            need = prefill_workspace_bytes(d);
        else if (quant_prefill_eligible(*dc, d) && off >= quant_prefill_workspace_bytes(d))
            need = 0;  // the tensor-core prefill, whose workspace fits
        if (need > off) return QG_ERR_WORKSPACE;
        cudaError_t e = cudaMemcpyAsync(xs, a.x, xb, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e);
        rc = run_gemv(d, call_ws, off, stream);
        if (rc) return rc;
        for (int i = 0; i < a.nw; ++i) {
            e = cudaMemcpyAsync(a.y[i], ys[i], yb, cudaMemcpyDeviceToHost, s);
            if (e != cudaSuccess) return cuda_fail(e);
        }
    }
    const cudaError_t e = cudaStreamSynchronize(s);
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

}  // namespace

int q4_k_cuda_core(const void* w, const float* x, float* y, int64_t M, int64_t N, int64_t K,
                   void* ws, size_t ws_bytes, qg_stream_t stream) {
    GemvArgs a{};
    a.fmt = FMT_Q4_K;
    a.nw = 1;
    a.w[0] = static_cast<const uint8_t*>(w);
    a.y[0] = y;
    a.x = x;
    a.M = M; a.N = N; a.K = K;
    int rc = validate_gemv(a);
    if (rc) return rc;
    if (ws && !aligned(ws, 16)) return QG_ERR_MISALIGNED;
    const DevCtx* dc = nullptr;
    rc = current_ctx(&dc);
    if (rc) return rc;
    if (gemv_workspace_bytes(*dc, a) > (ws ? ws_bytes : 0)) return QG_ERR_WORKSPACE;
    return gemv_launch(*dc, a, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

long long launch_option(int option) {
    switch (option) {
        case QG_OPT_PDL: return g_opt_pdl.load(std::memory_order_relaxed);
        case QG_OPT_PREFILL_MIN_M: return g_opt_prefill_min_m.load(std::memory_order_relaxed);
        case QG_OPT_STREAM: return g_opt_stream.load(std::memory_order_relaxed);
        case QG_OPT_STREAM_WARPS: return g_opt_stream_warps.load(std::memory_order_relaxed);
        case QG_OPT_STREAM_SLOTS: return g_opt_stream_slots.load(std::memory_order_relaxed);
        case QG_OPT_STAGES_AHEAD: return g_opt_ahead.load(std::memory_order_relaxed);
        case QG_OPT_STAGED_WARPS: return g_opt_staged_warps.load(std::memory_order_relaxed);
        case QG_OPT_PREFILL_FOLD: return g_opt_prefill_fold.load(std::memory_order_relaxed);
        case QG_OPT_XREG: return g_opt_xreg.load(std::memory_order_relaxed);
        case QG_OPT_XREG_AHEAD: return g_opt_xreg_ahead.load(std::memory_order_relaxed);
        case QG_OPT_XREG_WARPS: return g_opt_xreg_warps.load(std::memory_order_relaxed);
        case QG_OPT_XREG_CTAS: return g_opt_xreg_ctas.load(std::memory_order_relaxed);
        default: return 0;
    }
}

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return QG_ERR_CUDA;
}

// Workspace bytes of op; with quant_prefill the Q4_0 / Q4_K tensor-core
// prefill is included.
int workspace_size_impl(int op, int64_t M, int64_t N, int64_t K, int group_size, int packed,
                        size_t* bytes, bool quant_prefill) {
    if (!bytes) return QG_ERR_INVALID_ARG;
    *bytes = 0;
    if (op == QG_OP_AF4_G64) {  // no workspace
        int rc = check_dims(M, N, K);
        if (rc) return rc;
        return (M > 32 || N % 64 || K % 64) ? QG_ERR_INVALID_ARG : QG_OK;
    }
    GemvArgs a{};
    switch (op) {
        case QG_OP_Q4_0: a.fmt = FMT_Q4_0; a.nw = 1; break;
        case QG_OP_DUAL_Q4_0: a.fmt = FMT_Q4_0; a.nw = 2; break;
        case QG_OP_DUAL_Q4_0_HOST: a.fmt = FMT_Q4_0; a.nw = 2; break;
        case QG_OP_Q4_K: a.fmt = FMT_Q4_K; a.nw = 1; break;
        case QG_OP_AFFINE:
            if (packed != 0 && packed != 1) return QG_ERR_INVALID_ARG;
            a.fmt = packed ? FMT_AFF_PACKED : FMT_AFF_U8;
            a.nw = 1;
            a.gs = group_size;
            break;
        default: return QG_ERR_INVALID_ARG;
    }
    int rc = check_dims(M, N, K);
    if (rc) return rc;
    a.M = M; a.N = N; a.K = K;
    // Plan with 16-byte aligned stand-in pointers: the size assumes the
    // caller's buffers allow the fastest path (an upper bound otherwise).
    static const uint8_t probe[16] __attribute__((aligned(16))) = {0};
    a.w[0] = a.w[1] = probe;
    a.scales = a.biases = a.x = reinterpret_cast<const float*>(probe);
    const DevCtx* dc = nullptr;
    rc = current_ctx(&dc);
    if (rc) return rc;
    *bytes = gemv_workspace_bytes(*dc, a);
    if (prefill_eligible(*dc, a)) *bytes = std::max(*bytes, prefill_workspace_bytes(a));
    if (quant_prefill && quant_prefill_eligible(*dc, a))
        *bytes = std::max(*bytes, quant_prefill_workspace_bytes(a));
    if (op == QG_OP_DUAL_Q4_0_HOST) *bytes = host_stage_offset(*bytes) + host_stage_bytes(a);
    return QG_OK;
}

int cuda_core_workspace_size(int op, int64_t M, int64_t N, int64_t K, size_t* bytes) {
    return workspace_size_impl(op, M, N, K, 0, 0, bytes, false);
}

}  // namespace qg

using namespace qg;

extern "C" {

int qgemv_q4_0(const void* w, const float* x, float* y, int64_t M, int64_t N, int64_t K,
               void* workspace, size_t workspace_bytes, qg_stream_t stream) {
    GemvArgs a{};
    a.fmt = FMT_Q4_0;
    a.nw = 1;
    a.w[0] = static_cast<const uint8_t*>(w);
    a.y[0] = y;
    a.x = x;
    a.M = M; a.N = N; a.K = K;
    return run_gemv(a, workspace, workspace_bytes, stream);
}

int qgemv_dual_q4_0(const void* w_a, const void* w_b, const float* x, float* y_a, float* y_b,
                    int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                    qg_stream_t stream) {
    GemvArgs a{};
    a.fmt = FMT_Q4_0;
    a.nw = 2;
    a.w[0] = static_cast<const uint8_t*>(w_a);
    a.w[1] = static_cast<const uint8_t*>(w_b);
    a.y[0] = y_a;
    a.y[1] = y_b;
    a.x = x;
    a.M = M; a.N = N; a.K = K;
    return run_gemv(a, workspace, workspace_bytes, stream);
}

int qgemv_dual_q4_0_host(const void* w_a, const void* w_b, const float* x, float* y_a,
                         float* y_b, int64_t M, int64_t N, int64_t K, void* workspace,
                         size_t workspace_bytes, qg_stream_t stream) {
    GemvArgs a{};
    a.fmt = FMT_Q4_0;
    a.nw = 2;
    a.w[0] = static_cast<const uint8_t*>(w_a);
    a.w[1] = static_cast<const uint8_t*>(w_b);
    a.y[0] = y_a;
    a.y[1] = y_b;
    a.x = x;
    a.M = M; a.N = N; a.K = K;
    return run_gemv_host(a, workspace, workspace_bytes, stream);
}

int qgemv_q4_k(const void* w, const float* x, float* y, int64_t M, int64_t N, int64_t K,
               void* workspace, size_t workspace_bytes, qg_stream_t stream) {
    GemvArgs a{};
    a.fmt = FMT_Q4_K;
    a.nw = 1;
    a.w[0] = static_cast<const uint8_t*>(w);
    a.y[0] = y;
    a.x = x;
    a.M = M; a.N = N; a.K = K;
    return run_gemv(a, workspace, workspace_bytes, stream);
}

int qmm_affine(const float* x, const void* q, const float* scales, const float* biases, float* y,
               int64_t M, int64_t N, int64_t K, int group_size, int packed, void* workspace,
               size_t workspace_bytes, qg_stream_t stream) {
    if (packed != 0 && packed != 1) return QG_ERR_INVALID_ARG;
    GemvArgs a{};
    a.fmt = packed ? FMT_AFF_PACKED : FMT_AFF_U8;
    a.nw = 1;
    a.w[0] = static_cast<const uint8_t*>(q);
    a.y[0] = y;
    a.x = x;
    a.scales = scales;
    a.biases = biases;
    a.gs = group_size;
    a.M = M; a.N = N; a.K = K;
    return run_gemv(a, workspace, workspace_bytes, stream);
}

int qg_prepare_af4_g64(const uint8_t* codes, const uint16_t* scales_bf16,
                       const uint16_t* biases_bf16, uint32_t* plane, uint32_t* metadata,
                       int64_t N, int64_t K, qg_stream_t stream) {
    if (!codes || !scales_bf16 || !biases_bf16 || !plane || !metadata) return QG_ERR_INVALID_ARG;
    int rc = check_dims(1, N, K);
    if (rc) return rc;
    if (N % 64 || K % 64) return QG_ERR_INVALID_ARG;
    if (!aligned(scales_bf16, 2) || !aligned(biases_bf16, 2) || !aligned(plane, 16) ||
        !aligned(metadata, 4))
        return QG_ERR_MISALIGNED;
    const DevCtx* dc = nullptr;
    rc = current_ctx(&dc);
    if (rc) return rc;
    return af4_prepare_launch(*dc, codes, scales_bf16, biases_bf16, plane, metadata, N, K,
                              reinterpret_cast<cudaStream_t>(stream));
}

int qmm_af4_g64(const float* x, const uint32_t* plane, const uint32_t* metadata, float* y,
                int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                qg_stream_t stream) {
    (void)workspace;
    (void)workspace_bytes;
    if (!x || !plane || !metadata || !y) return QG_ERR_INVALID_ARG;
    int rc = check_dims(M, N, K);
    if (rc) return rc;
    if (M > 32 || N % 64 || K % 64) return QG_ERR_INVALID_ARG;
    if (!aligned(x, 4) || !aligned(y, 4) || !aligned(plane, 16) || !aligned(metadata, 4))
        return QG_ERR_MISALIGNED;
    const long long yb = M * N * 4;
    if (overlap(y, yb, x, M * K * 4) || overlap(y, yb, plane, N * K / 2) ||
        overlap(y, yb, metadata, N * (K / 64) * 4))
        return QG_ERR_INVALID_ARG;
    const DevCtx* dc = nullptr;
    rc = current_ctx(&dc);
    if (rc) return rc;
    return af4_gemv_launch(*dc, x, plane, metadata, y, M, N, K,
                           reinterpret_cast<cudaStream_t>(stream));
}

int qkv_split(const float* qkv, float* q, float* k, float* v, int64_t seq, int64_t q_sp,
              int64_t k_sp, int64_t v_sp, qg_stream_t stream) {
    if (!qkv || !q || !k || !v) return QG_ERR_INVALID_ARG;
    if (seq <= 0 || q_sp <= 0 || k_sp <= 0 || v_sp <= 0) return QG_ERR_INVALID_ARG;
    const long long lim = 0x3FFFFFFFFFFFFFFFLL / 4;
    if (q_sp > lim - k_sp || q_sp + k_sp > lim - v_sp) return QG_ERR_INVALID_ARG;
    const long long ch = q_sp + k_sp + v_sp;
    if (seq > lim / ch) return QG_ERR_INVALID_ARG;
    if (!aligned(qkv, 4) || !aligned(q, 4) || !aligned(k, 4) || !aligned(v, 4))
        return QG_ERR_MISALIGNED;
    const long long in_b = seq * ch * 4;
    const float* outs[3] = {q, k, v};
    const long long ob[3] = {seq * q_sp * 4, seq * k_sp * 4, seq * v_sp * 4};
    for (int i = 0; i < 3; ++i) {
        if (overlap(outs[i], ob[i], qkv, in_b)) return QG_ERR_INVALID_ARG;
        for (int j = i + 1; j < 3; ++j)
            if (overlap(outs[i], ob[i], outs[j], ob[j])) return QG_ERR_INVALID_ARG;
    }
    const DevCtx* dc = nullptr;
    int rc = current_ctx(&dc);
    if (rc) return rc;
    return qkv_split_launch(*dc, qkv, q, k, v, seq, q_sp, k_sp, v_sp,
                            reinterpret_cast<cudaStream_t>(stream));
}

static int run_dequant(int fmt, const void* w, const float* s, const float* b, float* out,
                       int64_t N, int64_t K, int gs, qg_stream_t stream) {
    if (!w || !out) return QG_ERR_INVALID_ARG;
    int rc = check_dims(1, N, K);
    if (rc) return rc;
    if (fmt == FMT_Q4_0 && K % 32) return QG_ERR_INVALID_ARG;
    if (fmt == FMT_Q4_K && K % 256) return QG_ERR_INVALID_ARG;
    if (fmt == FMT_AFF_U8 || fmt == FMT_AFF_PACKED) {
        if (!s || !b) return QG_ERR_INVALID_ARG;
        if (gs < 2 || gs > 1024 || (gs & (gs - 1)) || K % gs) return QG_ERR_INVALID_ARG;
        if (fmt == FMT_AFF_PACKED && (K & 1)) return QG_ERR_INVALID_ARG;
        if (!aligned(s, 4) || !aligned(b, 4)) return QG_ERR_MISALIGNED;
    }
    if (!aligned(out, 4)) return QG_ERR_MISALIGNED;
    if (overlap(out, N * K * 4, w, weight_bytes(fmt, N, K))) return QG_ERR_INVALID_ARG;
    const DevCtx* dc = nullptr;
    rc = current_ctx(&dc);
    if (rc) return rc;
    return dequant_launch(*dc, fmt, static_cast<const uint8_t*>(w), s, b, out, N, K, gs,
                          reinterpret_cast<cudaStream_t>(stream));
}

int dequant_q4_0(const void* w, float* out, int64_t N, int64_t K, qg_stream_t stream) {
    return run_dequant(FMT_Q4_0, w, nullptr, nullptr, out, N, K, 0, stream);
}

int dequant_q4_k(const void* w, float* out, int64_t N, int64_t K, qg_stream_t stream) {
    return run_dequant(FMT_Q4_K, w, nullptr, nullptr, out, N, K, 0, stream);
}

int dequant_affine(const void* q, const float* scales, const float* biases, float* out,
                   int64_t N, int64_t K, int group_size, int packed, qg_stream_t stream) {
    if (packed != 0 && packed != 1) return QG_ERR_INVALID_ARG;
    return run_dequant(packed ? FMT_AFF_PACKED : FMT_AFF_U8, q, scales, biases, out, N, K,
                       group_size, stream);
}

int qg_workspace_size(int op, int64_t M, int64_t N, int64_t K, int group_size, int packed,
                      size_t* bytes) {
    return qg::workspace_size_impl(op, M, N, K, group_size, packed, bytes, true);
}


int qg_set_option(int option, int64_t value) {
    switch (option) {
        case QG_OPT_PDL:
            if (value < 0 || value > 2) return QG_ERR_INVALID_ARG;
            g_opt_pdl.store(value, std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_PREFILL_MIN_M:
            if (value < 1) return QG_ERR_INVALID_ARG;
            g_opt_prefill_min_m.store(value, std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_STREAM:
            if (value < 0 || value > 2) return QG_ERR_INVALID_ARG;
            g_opt_stream.store(value, std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_STREAM_WARPS:
            if (value < 0 || value > 8) return QG_ERR_INVALID_ARG;
            g_opt_stream_warps.store(value, std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_STREAM_SLOTS:
            if (value != 0 && (value < 2 || value > 8)) return QG_ERR_INVALID_ARG;
            g_opt_stream_slots.store(value, std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_STAGES_AHEAD:
            if (value < 0 || value > 64) return QG_ERR_INVALID_ARG;
            g_opt_ahead.store(value, std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_STAGED_WARPS:
            if (value != 0 && value != 8) return QG_ERR_INVALID_ARG;
            g_opt_staged_warps.store(value, std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_PREFILL_FOLD:
            if (value != 0 && value != 1) return QG_ERR_INVALID_ARG;
            g_opt_prefill_fold.store(value, std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_XREG:
            if (value != 0 && value != 1) return QG_ERR_INVALID_ARG;
            g_opt_xreg.store(value, std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_XREG_AHEAD:
            if (value < 0 || value > 16) return QG_ERR_INVALID_ARG;
            g_opt_xreg_ahead.store(value, std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_XREG_WARPS:
            if (value != 0 && value != 4 && value != 8 && value != 16) return QG_ERR_INVALID_ARG;
            g_opt_xreg_warps.store(value, std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_XREG_CTAS:
            if (value < 0 || value > 4) return QG_ERR_INVALID_ARG;
            g_opt_xreg_ctas.store(value, std::memory_order_relaxed);
            return QG_OK;
        default: return QG_ERR_INVALID_ARG;
    }
}

int qg_get_option(int option, int64_t* value) {
    if (!value) return QG_ERR_INVALID_ARG;
    switch (option) {
        case QG_OPT_PDL: *value = g_opt_pdl.load(std::memory_order_relaxed); return QG_OK;
        case QG_OPT_PREFILL_MIN_M:
            *value = g_opt_prefill_min_m.load(std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_STREAM: *value = g_opt_stream.load(std::memory_order_relaxed); return QG_OK;
        case QG_OPT_STREAM_WARPS:
            *value = g_opt_stream_warps.load(std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_STREAM_SLOTS:
            *value = g_opt_stream_slots.load(std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_STAGES_AHEAD: *value = g_opt_ahead.load(std::memory_order_relaxed); return QG_OK;
        case QG_OPT_STAGED_WARPS:
            *value = g_opt_staged_warps.load(std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_PREFILL_FOLD:
            *value = g_opt_prefill_fold.load(std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_XREG: *value = g_opt_xreg.load(std::memory_order_relaxed); return QG_OK;
        case QG_OPT_XREG_AHEAD:
            *value = g_opt_xreg_ahead.load(std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_XREG_WARPS:
            *value = g_opt_xreg_warps.load(std::memory_order_relaxed);
            return QG_OK;
        case QG_OPT_XREG_CTAS:
            *value = g_opt_xreg_ctas.load(std::memory_order_relaxed);
            return QG_OK;
        default: return QG_ERR_INVALID_ARG;
    }
}

const char* qg_status_string(int status) {
    switch (status) {
        case QG_OK: return "ok";
        case QG_ERR_INVALID_ARG: return "invalid argument";
        case QG_ERR_UNSUPPORTED: return "unsupported request";
        case QG_ERR_MISALIGNED: return "misaligned pointer";
        case QG_ERR_CUDA: return "CUDA runtime error";
        case QG_ERR_WORKSPACE: return "workspace missing or too small";
        case QG_ERR_DEVICE: return "a kernel reported an error";
        default: return "unknown status";
    }
}

int qg_last_cuda_error(void) { return t_last_cuda_error; }

int qg_device_error(int clear, unsigned int* code) {
    const DevCtx* dc = nullptr;
    int rc = current_ctx(&dc);
    if (rc) return rc;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
    if (e != cudaSuccess) return cuda_fail(e);
    if (clear && v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (code) *code = v;
    return v ? QG_ERR_DEVICE : QG_OK;
}

int qg_selftest_wait_timeout(int64_t timeout_ns, qg_stream_t stream) {
    if (timeout_ns <= 0) return QG_ERR_INVALID_ARG;
    if (timeout_ns > 2000000000LL) timeout_ns = 2000000000LL;
    const DevCtx* dc = nullptr;
    int rc = current_ctx(&dc);
    if (rc) return rc;
    return selftest_wait_launch(*dc, timeout_ns, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
