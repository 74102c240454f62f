// Shared pieces of the two tensor-core prefill kernels of qmm_affine
// (prefill.cu: exact integer codes, the default; prefill_fold.cu: weights
// folded to fp16): tile geometry, PTX wrappers for TMA, tcgen05 and tensor
// memory, warp-wide bounded barrier waits, and the folded kernel's entry.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "qg_internal.cuh"

namespace qg {
namespace prefill {

constexpr int kTileN = 128;    // weight rows per CTA (MMA M)
constexpr int kTileT = 128;    // activation rows per CTA (MMA N)
constexpr int kChunk = 64;     // k per stage (one 128-byte fp16 row)
constexpr int kTmemCols = 512;
constexpr int kXhBytes = kTileT * kChunk * 2;  // 16 KB per stage
constexpr int kPrepThreads = 256;

// Stage geometry shared by both kernels: a 64-wide k chunk of the code tile
// (u8: 64 bytes per row, packed: 32) after the 16 KB fp16 x tile.
template <bool PACKED>
struct StageGeo {
    static constexpr int kCodeRowBytes = PACKED ? kChunk / 2 : kChunk;    // per stage
    static constexpr int kCodeBytes = kTileN * kCodeRowBytes;
    static constexpr int kStageBytes = kXhBytes + kCodeBytes;             // multiple of 1024
};

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// 1-D bulk copy global -> shared without a cache hint (data many CTAs read).
__device__ __forceinline__ void bulk_g2s_nohint(uint32_t dst, const void* src, uint32_t bytes,
                                                uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]; fp16 inputs, f32 accumulate.
__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 16 consecutive 32-bit columns of this thread's lane, waited on in the same
// statement so no use of the registers can be scheduled before the data.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Issue a 16-column load without waiting; tmem_wait16 completes it. The
// registers pass through the wait as read-write operands, so no use of them
// can be scheduled between the two.
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand in 128-byte swizzle atoms
// (8 rows x 128 bytes, atoms 1024 bytes apart), start address in 16-byte units.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) |
           (2ull << 61);
}

// Instruction descriptor, kind::f16: f32 accumulator, fp16 A and B, both
// K-major, N = kTileT, M = kTileN.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kTileT >> 3) << 17) | ((uint32_t)(kTileN >> 4) << 24);

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity);
    return __all_sync(0xFFFFFFFFu, ok);
}

// warp_wait for warps that run ahead of the MMA issuer (fold_kernel's
// converters): suspended while waiting, so that they do not take issue
// slots from the one thread that issues the MMAs.
__device__ __forceinline__ bool warp_wait_sleep(uint32_t bar, uint32_t parity) {
    const bool ok = mbar_wait_sleep(bar, parity);
    return __all_sync(0xFFFFFFFFu, ok);
}

struct FoldParams {
    const float* scales_t;  // [G, N]
    const float* biases_t;  // [G, N]
    const float* bpart;     // [N, GT] max_g (|s| * qmax + |b|) over 32-group tiles
    const float* inv;       // [Mp] 2^-e_m
    float* y;               // [M, N]
    int M, N, K, G, GT;
    int log2gs;
    unsigned* err;
};

// Launch of fold_kernel<packed, gs == 16> (prefill_fold.cu) as a programmatic
// dependent of the prep kernel, and its dynamic shared memory bytes.
int launch_fold_kernel(const DevCtx& dc, bool packed, bool gs16, const CUtensorMap& mq,
                       const CUtensorMap& mx, const FoldParams& fp, dim3 grid, cudaStream_t s);
int fold_smem_bytes(bool packed);

// cuTensorMapEncodeTiled from the driver, looked up once (prefill.cu).
int encoder(PFN_cuTensorMapEncodeTiled_v12000* out);

}  // namespace prefill
}  // namespace qg
