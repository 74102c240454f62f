/*
 * qgemv.h - C ABI of libqgemv.so: quantized matrix-vector and skinny matmul
 * with fused dequantization, for NVIDIA GB300 (sm_103a).
 *
 *   y[M, N] = x[M, K] . dequant(W)[N, K]^T      (f32 in, f32 out)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All pointers are DEVICE pointers owned by the caller; the library keeps
 *   none of them after the call returns. Row-major, densely packed.
 * - Calls are asynchronous: they enqueue work on `stream` (NULL = the legacy
 *   default stream) and return. Results are valid once the stream is
 *   synchronized. Nothing is allocated on the device by these calls.
 * - Every call validates its arguments first; on a validation failure it
 *   enqueues nothing and returns a non-zero qg_status. A failed launch
 *   returns QG_ERR_CUDA (qg_last_cuda_error() gives the cudaError_t).
 * - Buffer lengths cannot be checked through raw pointers: the sizes stated
 *   below are preconditions. Outputs must not overlap inputs or each other.
 * - Alignment: x, y, scales and biases need 4-byte alignment (else
 *   QG_ERR_MISALIGNED); weights may start at any byte.
 *   The fastest path additionally wants 16-byte aligned weight rows
 *   (K % 256 == 0 and 16-byte aligned base pointers); otherwise a slower
 *   general kernel computes the same result within the same tolerance.
 * - Accuracy: every f32 output y satisfies |y - ref| <= 1e-5 * B + 1e-6 where
 *   ref is the exact dot product of x with the dequantized weights and
 *   B = sum_k |x_k w_k| (the tensor-core prefill path: 2e-3 * B + 1e-6).
 *   Dequantization exports are bit-exact.
 * - Workspace: the GEMV/qmm calls may need device scratch for a deterministic
 *   split-K reduction or a prefill prologue. Query the size with
 *   qg_workspace_size(); pass a buffer at least that large (16-byte aligned),
 *   or NULL/0 when the size is 0. Too small a buffer returns
 *   QG_ERR_WORKSPACE. Calls that share one workspace must not overlap.
 *
 * Formats
 * -------
 * Q4_0   (page: fused_dual_proj_q4_0.rs, mlx-native 0.9.1, preconditions of
 *        dispatch_fused_dual_proj_q4_0): 32 weights per 18-byte block, fp16 d
 *        (little-endian) then 16 bytes; byte 2+j holds element j in its low
 *        nibble and element 16+j in its high nibble; w = (q - 8) * d. Weight
 *        matrix = N rows of K/32 blocks. Requires K % 32 == 0.
 * Q4_K   (page: q4_k_gemv_v2.rs, ferrum-kernels 0.7.7, module doc):
 *        256 weights per 144-byte super-block: fp16 d, fp16 dmin, 12 bytes of
 *        packed 6-bit (scale, min) pairs for 8 sub-blocks of 32, 128 nibble
 *        bytes (chunk c of 32 bytes: low nibbles = sub-block 2c, high nibbles
 *        = sub-block 2c+1); w = (d*sc)*q - dmin*m. N rows of K/256
 *        super-blocks. Requires K % 256 == 0.
 * affine (page: qmm_affine.rs, mlx-native 0.21.1, qmm_affine_t_cpu and
 *        pack_b4_to_u32): w[n,k] = fma(q[n,k], s[n,g], b[n,g]), g = k / gs,
 *        gs a power of two in [2, 1024], K % gs == 0. Codes are one u8 per
 *        element ([N, K] bytes, packed = 0) or two 4-bit codes per byte
 *        ([N, K/2] bytes, element 2i in the low nibble of byte i, packed = 1,
 *        K even). s, b: f32 [N, K/gs].
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define QG_API __attribute__((visibility("default")))
#else
#define QG_API
#endif

/* Same type as cudaStream_t; declared here so that this header needs no CUDA
 * header. */
typedef struct CUstream_st* qg_stream_t;

typedef enum {
    QG_OK = 0,
    QG_ERR_INVALID_ARG = 1,   /* zero/negative dims, bad divisibility, NULL, aliasing */
    QG_ERR_UNSUPPORTED = 2,   /* valid request outside what this build supports */
    QG_ERR_MISALIGNED = 3,    /* pointer alignment below the stated minimum */
    QG_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    QG_ERR_WORKSPACE = 5,     /* workspace missing or smaller than required */
    QG_ERR_DEVICE = 6         /* a kernel reported an error (see qg_device_error) */
} qg_status;

/* Operation ids for qg_workspace_size. */
enum {
    QG_OP_Q4_0 = 0,
    QG_OP_DUAL_Q4_0 = 1,
    QG_OP_Q4_K = 2,
    QG_OP_AFFINE = 3,
    QG_OP_AF4_G64 = 4,
    QG_OP_DUAL_Q4_0_HOST = 5  /* qgemv_dual_q4_0_host: the call's own workspace plus
                                 device staging for x, y_a, y_b */
};

/* Single Q4_0 projection: y[M,N] = x[M,K] . dequant(w)[N,K]^T.
 * Page: fused_dual_proj_q4_0.rs (mlx-native 0.9.1) - the baseline
 * kernel_mul_mv_q4_0_f32 dispatch the fused op is defined against.
 * w: N*(K/32)*18 bytes; x: M*K f32; y: M*N f32. M, N, K > 0, K % 32 == 0.
 *
 * Q4_0 and Q4_K calls take one of two paths:
 * - CUDA cores, f32 (|y - exact| <= 1e-5 * sum_k |x w| + 1e-6), for every M.
 * - Tensor cores (prefill), when M >= QG_OPT_PREFILL_MIN_M (default 64), x is
 *   16-byte aligned, the tensor-core prefill conditions of qmm_affine hold for
 *   group size 32, and the workspace is at least qg_workspace_size bytes. The
 *   weights are rewritten in the workspace as packed affine codes per 32
 *   weights (Q4_0: scale d, bias -8d; Q4_K: scale d*sc, bias -dmin*m, all
 *   exact) and multiplied as qmm_affine's prefill does; the error bound is
 *   qmm_affine's (2e-3 * sum_k |x w|). A smaller workspace (as small as the
 *   CUDA-core path needs) keeps the call on CUDA cores. */
QG_API int qgemv_q4_0(const void* w, const float* x, float* y, int64_t M, int64_t N, int64_t K,
               void* workspace, size_t workspace_bytes, qg_stream_t stream);

/* Fused dual Q4_0 projection: two weights of equal shape share one input.
 * Page: fused_dual_proj_q4_0.rs (mlx-native 0.9.1), dispatch_fused_dual_proj_q4_0
 * ("byte-identical to two kernel_mul_mv_q4_0_f32 dispatches").
 * y_a = x . dequant(w_a)^T, y_b = x . dequant(w_b)^T; each output is bitwise
 * equal to what qgemv_q4_0 returns for the same weight when both weights
 * take the same path (same alignment class). Sizes as for qgemv_q4_0;
 * y_a != y_b. */
QG_API int qgemv_dual_q4_0(const void* w_a, const void* w_b, const float* x, float* y_a, float* y_b,
                    int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                    qg_stream_t stream);

/* qgemv_dual_q4_0 with x, y_a and y_b in HOST memory; w_a and w_b stay in
 * device memory (model weights are resident). The operation is the page's
 * (fused_dual_proj_q4_0.rs, dispatch_fused_dual_proj_q4_0); taking host
 * buffers and returning only when the result is in them is this library's
 * own addition, for callers whose input arrives from, and whose output goes
 * back to, the host every step (the host round trip qkv_split.rs's module
 * doc names as the cost to cut).
 * - Synchronous: returns after y_a and y_b hold the result (it synchronizes
 *   `stream`, so work queued on it earlier completes first). Results equal
 *   qgemv_dual_q4_0's on device copies of the same buffers, bit for bit.
 * - Zero-copy: when x, y_a and y_b are page-locked host memory mapped for the
 *   device (cudaHostAlloc, or cudaHostRegister with cudaHostRegisterMapped),
 *   x is 16-byte aligned, and every slice of the call runs on the
 *   register-resident-x kernel (M <= 2 for this format), a small kernel
 *   copies x from host memory into the workspace and the GEMV, launched as
 *   its programmatic dependent, reads x there and writes y_a and y_b straight
 *   into host memory (plain stores over the host link). No copy-engine
 *   transfer is enqueued.
 * - Otherwise (pageable buffers, other M): x is copied into the workspace,
 *   the call runs there and y_a, y_b are copied back, each with one
 *   cudaMemcpyAsync on `stream`.
 * - workspace: device memory of at least
 *   qg_workspace_size(QG_OP_DUAL_Q4_0_HOST, M, N, K, 0, 0) bytes, 16-byte
 *   aligned, on both routes (the staging of x, y_a and y_b sits at its end);
 *   QG_ERR_WORKSPACE (nothing enqueued) when it is smaller.
 * - Host buffers must not overlap one another. Errors as for
 *   qgemv_dual_q4_0; a failed copy or synchronization returns QG_ERR_CUDA. */
QG_API int qgemv_dual_q4_0_host(const void* w_a, const void* w_b, const float* x, float* y_a,
                                float* y_b, int64_t M, int64_t N, int64_t K, void* workspace,
                                size_t workspace_bytes, qg_stream_t stream);

/* Q4_K GEMV. Page: q4_k_gemv_v2.rs (ferrum-kernels 0.7.7),
 * dispatch_gemv_q4k_v2_offset (M = 1 there; any M here; the two paths of
 * qgemv_q4_0 apply).
 * w: N*(K/256)*144 bytes; x: M*K f32; y: M*N f32. K % 256 == 0. Callers that
 * keep several tensors in one buffer pass offset pointers (byte offsets
 * must keep the stated alignment). */
QG_API int qgemv_q4_k(const void* w, const float* x, float* y, int64_t M, int64_t N, int64_t K,
               void* workspace, size_t workspace_bytes, qg_stream_t stream);

/* qgemv_q4_k for callers that cannot call cudaMalloc (code inside someone
 * else's CUDA graph capture, plugins whose host application owns every device
 * allocation, runtimes that forbid allocation after start-up). No counterpart
 * in the source pages: an addition of this library. Same arguments, result
 * and accuracy as qgemv_q4_k, but the split-K scratch that qgemv_q4_k takes
 * as a workspace comes from a 4 MiB array in the library's own device memory
 * (held on every GPU that loads the library until the process exits).
 * - Returns QG_ERR_WORKSPACE, before enqueuing anything, when the CUDA-core
 *   kernels need more than 4 MiB of split-K scratch for the shape (at most
 *   qg_workspace_size(QG_OP_Q4_K, ...), which also covers the prefill).
 * - Allocates nothing. The first call on a device looks up the array's device
 *   address (cudaGetSymbolAddress); make that first call before any stream
 *   capture. A failed lookup is not remembered: the next call tries again.
 * - All calls share the one array: calls that may overlap on the GPU (other
 *   streams, other host threads) race on it. Its contents are fully rewritten
 *   before they are read, so nothing needs clearing between calls.
 * - Always takes qgemv_q4_k's CUDA-core kernels, for every M, with their f32
 *   bound (1e-5 * sum_k |x w| + 1e-6): the tensor-core prefill needs scratch
 *   for the rewritten weights, which this entry point does not have. */
QG_API int qgemv_q4_k_noalloc(const void* w, const float* x, float* y, int64_t M, int64_t N,
                              int64_t K, qg_stream_t stream);

/* Affine group-quantized matmul y = x . dequant(q, s, b)^T.
 * Page: qmm_affine.rs (mlx-native 0.21.1), dispatch_qmm_affine_t_f32 and
 * dispatch_qmm_affine_t_packed_simd4_b4 (packed 4-bit codes). The packed and
 * one-code-per-byte storages give bitwise-identical y.
 *
 * Two paths, chosen per call:
 * - CUDA cores, f32 throughout (|y - exact| <= 1e-5 * sum_k |x w| + 1e-6):
 *   M below the QG_OPT_PREFILL_MIN_M option (default 64), or any of the
 *   tensor-core conditions below unmet.
 * - Tensor cores (prefill), when M >= QG_OPT_PREFILL_MIN_M, group_size >= 16,
 *   K % 16 == 0 (K % 32 == 0 when packed), q and x 16-byte aligned, M, N, K
 *   <= 2^30 and N <= 8,388,480. Each x row is scaled by a power of two and
 *   rounded to fp16 once; the codes enter the MMA as exact fp16 integers and
 *   per-group f32 partial sums get scale and bias in an f32 epilogue (the
 *   regrouping the page's bf16 table-plus-sums kernels use). Error:
 *   |y - exact| <= 2^-11 * sum_k |x w| plus f32 rounding; callers should
 *   budget 2e-3 * sum_k |x w|. Needs a workspace of qg_workspace_size bytes
 *   (the fp16 copy of x plus per-group sums).
 * Non-finite x propagates to the affected y rows on both paths. */
QG_API int qmm_affine(const float* x, const void* q, const float* scales, const float* biases, float* y,
               int64_t M, int64_t N, int64_t K, int group_size, int packed, void* workspace,
               size_t workspace_bytes, qg_stream_t stream);

/* Split a fused [seq, q_sp + k_sp + v_sp] f32 tensor into q [seq, q_sp],
 * k [seq, k_sp], v [seq, v_sp]. Page: qkv_split.rs (mlx-native 0.7.1),
 * dispatch_qkv_split_f32. A bit copy: every 32-bit word, NaN payloads
 * included, lands unchanged in exactly one output. All spans > 0; their sum
 * must not overflow. */
QG_API int qkv_split(const float* qkv, float* q, float* k, float* v, int64_t seq, int64_t q_sp,
              int64_t k_sp, int64_t v_sp, qg_stream_t stream);

/* Dequantize a whole weight matrix to f32 out[N, K], bit-exact with the
 * format definition. Page: qmm_affine.rs (mlx-native 0.21.1), the
 * qdq_affine forward composition test (dequantize, then matmul). */
QG_API int dequant_q4_0(const void* w, float* out, int64_t N, int64_t K, qg_stream_t stream);
QG_API int dequant_q4_k(const void* w, float* out, int64_t N, int64_t K, qg_stream_t stream);
QG_API int dequant_affine(const void* q, const float* scales, const float* biases, float* out,
                   int64_t N, int64_t K, int group_size, int packed, qg_stream_t stream);

/* The prepared 4-bit affine layout with groups of 64 ("AF4-g64").
 * Page: qmm_affine.rs (mlx-native 0.21.1), prepare_af4_g64 (test module) and
 * dispatch_qmm_affine_t_packed_simd4_b4_gs64_bf16. N % 64 == 0, K % 64 == 0.
 *  - plane: u32 [N/64][K/32][64][4]. Word c (0..3) of (row r, 32-group g)
 *    holds codes of row r at k = 32g + e: for pair p = 0..3, with
 *    e0 = 16 (p >> 1) + 4c + 2 (p & 1), code e0 in bits 4p..4p+3 and code
 *    e0 + 1 in bits 16 + 4p..19 + 4p.
 *  - metadata: u32 [N/64][K/64][64]: bf16 scale | bf16 bias << 16 of
 *    (row, 64-group).
 * The weight is w = scale * q + bias, with the bf16 values taken exactly as
 * f32 and one f32 rounding (as qmm_affine).
 *
 * qg_prepare_af4_g64 writes plane and metadata from codes (u8 [N, K], values
 * 0..15) and the bf16 bits of scales and biases (u16 [N, K/64]). A bit
 * rearrangement: the result is exact.
 *
 * qmm_af4_g64: y[M,N] = x[M,K] . w[N,K]^T from the prepared layout, M <= 32
 * (the page's limit). The page's kernel rounds x to bf16 (error class:
 * relative RMS and max |err| / max(|y|, 1) <= 5e-3). Here the kernels read
 * the prepared words directly and compute in f32 on the CUDA cores for
 * every M: |y - exact| <= 1e-5 * sum_k |x w| + 1e-6. M = 1 and 2 take the
 * register-resident-x kernel when K <= 4096 (K <= 1024, 2048 or 4096 of
 * whole warps of 32-groups: K in (2048, 3072] excluded) and x, plane and
 * metadata are 16-byte aligned; other calls a kernel that splits K across a
 * thread-block cluster. Row m of y is bitwise the same for M = 1 and 2, for
 * every M in 3..8 and for every M in 9..32. x and y 4-byte aligned, plane 16-byte aligned,
 * metadata 4-byte aligned; y must not overlap an input. No workspace
 * (qg_workspace_size reports 0; workspace may be NULL). */
QG_API int qg_prepare_af4_g64(const uint8_t* codes, const uint16_t* scales_bf16,
                              const uint16_t* biases_bf16, uint32_t* plane, uint32_t* metadata,
                              int64_t N, int64_t K, qg_stream_t stream);
QG_API int qmm_af4_g64(const float* x, const uint32_t* plane, const uint32_t* metadata, float* y,
                       int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                       qg_stream_t stream);

/* Workspace bytes op (QG_OP_*) needs for the given shape; *bytes = 0 when
 * none. group_size/packed matter only for QG_OP_AFFINE. Returns a status. */
QG_API int qg_workspace_size(int op, int64_t M, int64_t N, int64_t K, int group_size, int packed,
                      size_t* bytes);

/* Process-wide launch options (not a counterpart of anything on the pages;
 * they select how this library's kernels are launched).
 *
 * QG_OPT_PDL (default 0): 1 launches the GEMV/qmm kernels with programmatic
 * dependent launch. A kernel then starts while the previous kernel on the
 * stream is still draining and streams its weights right away; it waits for
 * the previous kernel to complete only before it reads x and writes y. The
 * caller promises that the weight codes, scales and biases of a call are not
 * written by the kernel immediately preceding it on the stream (static model
 * weights satisfy this). Back-to-back decode projections overlap one call's
 * ramp-up with the previous call's tail this way.
 *
 * QG_OPT_PDL = 2 adds a second promise: the call reads nothing the kernel
 * immediately preceding it on the stream writes, and writes nothing that
 * kernel reads or writes (independent projections, e.g. several projections
 * of one input, or calls on distinct buffers). The register-resident-x
 * kernel (QG_OPT_XREG) and the staged kernel (when the call needs no split-K
 * workspace, which consecutive calls may share) then do not wait for their
 * predecessor at all, so consecutive independent calls run concurrently; the
 * other kernels behave as with 1. A kernel launched after such a call
 * without programmatic dependent launch still waits for it as usual. */
/*
 * QG_OPT_PREFILL_MIN_M (default 64, >= 1): smallest M for which qmm_affine
 * (and the Q4_0 / Q4_K calls) take the tensor-core prefill path when its
 * other conditions hold. Below it every call keeps the f32 bound. */
/*
 * QG_OPT_STREAM (default 1): which GEMV/qmm calls with M <= 2 (per slice of
 * x) take the streaming kernel instead of the staged-stage kernel. 0: none.
 * 1: where it is the faster of the two (Q4_K, except two rows with
 * K > 8192). 2: every
 * eligible call. Eligible: K % 256 == 0, (K / 256) % 4 == 0, the weight, x
 * (and affine scale/bias) pointers 16-byte aligned and, for affine weights,
 * group_size >= 32. Both kernels give results within the same tolerance; the
 * choice never depends on N or on single versus dual calls, so the dual
 * projection stays bitwise equal to two single projections under any
 * setting.
 *
 * QG_OPT_STREAM_WARPS (default 0 = automatic; else 1..8) and
 * QG_OPT_STREAM_SLOTS (default 0 = automatic; else 2..8): warps per CTA and
 * shared-memory ring slots per warp of the streaming kernel (tuning). A
 * setting whose shared memory does not fit falls back to the automatic one. */
/*
 * QG_OPT_STAGES_AHEAD (default 2; 0 = every stage of the ring; else 1..64):
 * for M <= 2 (per slice of x) the staged-stage kernel requests weight chunk i
 * only once chunk i - n has landed, so that each SM's first chunks are not
 * queued behind the whole grid's traffic (tuning; a value above the ring size
 * means the ring size). */
/*
 * QG_OPT_STAGED_WARPS (default 0 = automatic; or 8): with 8, M = 1 calls of
 * the staged-stage kernel use eight consumer warps and at most half an SM's
 * registers and shared memory, so that the next launch's CTA can be resident
 * beside this one (tuning). */
/*
 * QG_OPT_PREFILL_FOLD (default 0; or 1): which tensor-core prefill kernel
 * qmm_affine (and the Q4_0/Q4_K prefill built on it) runs. 0: exact integer
 * codes on the tensor cores, scale and bias applied per group in an f32
 * epilogue. 1: scale and bias folded into fp16 weights,
 * w' = fp16((s q + b) 2^f_n) with a power of two per weight row, one f32
 * accumulator over all of K, faster. Both stay within 2e-3 * sum_k |x w|
 * for weight rows whose scales span less than 2^29; 0 keeps the weights
 * exact whatever their spread. */
/*
 * QG_OPT_XREG (default 1; or 0): calls with M <= 2 (per slice of x) take the
 * register-resident-x kernel when it is eligible: K % 32 == 0, K <= 16384,
 * Q4_0 rows 16-byte aligned (K % 256 == 0), affine group size >= 32 with
 * (K / group_size) % 4 == 0, and the weight, x (and affine scale / bias)
 * pointers 16-byte aligned. 0 leaves those calls to the other CUDA-core
 * kernels. Like QG_OPT_STREAM, the choice never depends on N or on single
 * versus dual calls.
 *
 * QG_OPT_XREG_AHEAD (default 0 = every slot of the ring; else 1..16): chunks
 * of weights the register-resident-x kernel keeps in flight at most (tuning).
 *
 * QG_OPT_XREG_WARPS (default 0 = automatic; or 4, 8, 16) and
 * QG_OPT_XREG_CTAS (default 0 = automatic; or 1..4): consumer warps per CTA
 * and CTAs per SM per call of the register-resident-x kernel (tuning;
 * results are bitwise the same). A count that does not suit the shape (the
 * warps of one row group must divide it; sixteen warps take one x row) falls
 * back to automatic. With four consumer warps (rows of at most 4096 weights
 * of K), four CTAs share an SM; automatic picks them when QG_OPT_PDL is 2,
 * eight warps otherwise and for the host-buffer call (a lone call, which
 * also takes all of the SM's shared memory). Automatic CTAs, when QG_OPT_PDL
 * is 2 and a slice has one or two rows of x (the calls' CTAs overlap): three
 * per four SMs per call for one row of x on four warps (one per two SMs for
 * qmm_af4_g64), one per two SMs for one row on more warps, one per four SMs
 * for two rows; one per SM in every other case. */
enum { QG_OPT_PDL = 1, QG_OPT_PREFILL_MIN_M = 2, QG_OPT_STREAM = 3, QG_OPT_STREAM_WARPS = 4,
       QG_OPT_STREAM_SLOTS = 5, QG_OPT_STAGES_AHEAD = 6, QG_OPT_STAGED_WARPS = 7,
       QG_OPT_PREFILL_FOLD = 8, QG_OPT_XREG = 9, QG_OPT_XREG_AHEAD = 10,
       QG_OPT_XREG_WARPS = 11, QG_OPT_XREG_CTAS = 12 };
QG_API int qg_set_option(int option, int64_t value);
QG_API int qg_get_option(int option, int64_t* value);

/* Human-readable text of a qg_status. Never NULL. */
QG_API const char* qg_status_string(int status);

/* cudaError_t of the most recent QG_ERR_CUDA on this host thread. */
QG_API int qg_last_cuda_error(void);

/* Kernels never trap: a kernel that gives up on a bounded wait records a
 * non-zero code in a per-device error word instead. This call synchronizes
 * the current device, reads the word into *code (may be NULL) and clears it
 * when clear != 0. Returns QG_OK, or QG_ERR_DEVICE when the word was
 * non-zero. */
QG_API int qg_device_error(int clear, unsigned int* code);

/* Self-test of the bounded wait: launches one block that waits on a barrier
 * nobody arrives at for about timeout_ns nanoseconds (capped at 2 s), then
 * records its timeout code in the device error word and exits. */
QG_API int qg_selftest_wait_timeout(int64_t timeout_ns, qg_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H */
