// qmm on the prepared AF4-g64 layout: y[M,N] = x[M,K] . w[N,K]^T, M <= 32,
// w = scale * q + bias per (row, 64-group), scale and bias bf16.
//
// Page: qmm_affine.rs (mlx-native 0.21.1): prepare_af4_g64 (layout) and
// dispatch_qmm_affine_t_packed_simd4_b4_gs64_bf16 (the call). The page's
// Metal kernel rounds x to bf16 and multiplies 8-row tiles on simdgroup
// matrices; here the arithmetic stays f32 on the CUDA cores. Design for
// sm_103a, read straight from the prepared layout:
//
//  * The plane keeps the 64 rows of a row block side by side per 32-group
//    (64 x 16 bytes = 1 KB contiguous). Lane l of a warp owns rows l and
//    l + 32 of the block, so each 16-byte load of a warp reads 512 contiguous
//    bytes, and no cross-lane reduction is needed for a row's dot product.
//  * Every lane needs the same x values: x is staged once per CTA in shared
//    memory and read back as warp-wide broadcasts (one float4 per word and
//    activation row, used for both of the lane's rows).
//  * Decode: nibble n of a word sits at bit 4n. (word & 0xF << 4n) | 0x4B000000
//    is the exact float 2^23 + q * 2^(4n) for n <= 4; nibbles 5..7 are taken
//    from the word shifted right by 12 (at 2^8, 2^12, 2^16). One packed f32x2
//    subtraction of 2^23 leaves q * 2^s exactly, and the staged x was
//    pre-multiplied by 2^-s, so each packed f32x2 FMA adds q * x with one
//    rounding (exact scaling for |x| >= 2^-110).
//  * Per (row, 64-group) the sum of q * x is kept in a float pair, then
//    scale * sum + bias * sum(x) is added to the warp's partial output. The
//    sums of x per 64-group are taken from the unscaled x.
//  * A CTA covers one row block and a K slice; warp w takes the slice's
//    64-groups w, w + 8, ... and prefetches its next group's words while it
//    computes the current one. The 8 warps' partials are added in warp
//    order, then the K slices of a row block (the CTAs of one thread-block
//    cluster) are added in cluster-rank order through distributed shared
//    memory. Each output's arithmetic is fixed by N, K, the SM count and
//    whether M <= 8 (which sets the number of K slices): it does not depend
//    on how many activation rows a tile takes or on how x is staged, so row
//    m of y is bitwise the same for every M in 1..8, and for every M in
//    9..32.
#include <algorithm>

#include "qg_internal.cuh"

namespace qg {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxKS = 8;
constexpr int kXB = 8;        // x loads in flight per thread while staging

struct Params {
    const float* x;
    const uint4* plane;      // 16-byte (row, 32-group) units
    const uint32_t* meta;
    float* y;
    int M, N, K;
    int G32, G64;
    int gpc;                 // 64-groups per CTA (K slice)
    int cap;                 // 64-groups per x sub-slice (a multiple of kWarps, or gpc)
    int KS;                  // K slices = CTAs per cluster
    uint32_t magic;          // 0x4B000000, passed in so it stays in a register
};

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Weight words are read once: no L1 allocation, evict first from L2.
__device__ __forceinline__ uint4 ld_stream(const uint4* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ uint32_t ld_stream(const uint32_t* p, uint64_t pol) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;"
                 : "=r"(v)
                 : "l"(p), "l"(pol));
    return v;
}

// (v & MASK) | mg in one LOP3.
template <uint32_t MASK>
__device__ __forceinline__ float and_or(uint32_t v, uint32_t mg) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(v), "n"(MASK), "r"(mg));
    return __uint_as_float(d);
}

// Word c of a (row, 32-group) unit -> four pairs of exact values q * 2^s,
// in element order: f[0] = codes (4c, 4c+1), f[1] = (4c+2, 4c+3),
// f[2] = (16+4c, 17+4c), f[3] = (18+4c, 19+4c) of the group.
__device__ __forceinline__ void decode(uint32_t v, uint32_t mg, float2 (&f)[4]) {
    const uint32_t v2 = v >> 12;
    const float2 c = make_float2(-8388608.0f, -8388608.0f);
    f[0] = __fadd2_rn(make_float2(and_or<0x0000Fu>(v, mg), and_or<0xF0000u>(v, mg)), c);
    f[1] = __fadd2_rn(make_float2(and_or<0x000F0u>(v, mg), and_or<0x00F00u>(v2, mg)), c);
    f[2] = __fadd2_rn(make_float2(and_or<0x00F00u>(v, mg), and_or<0x0F000u>(v2, mg)), c);
    f[3] = __fadd2_rn(make_float2(and_or<0x0F000u>(v, mg), and_or<0xF0000u>(v2, mg)), c);
}

// 2^-s for element j of a 32-group (s as decode leaves it): elements
// 4c + (0, 1, 2, 3) carry 2^(0, 16, 4, 8), elements 16 + 4c + (0..3) carry
// 2^(8, 12, 12, 16).
__device__ __forceinline__ float4 x_scale(int j) {
    return (j & 16) ? make_float4(1.0f / 256.0f, 1.0f / 4096.0f, 1.0f / 4096.0f, 1.0f / 65536.0f)
                    : make_float4(1.0f, 1.0f / 65536.0f, 1.0f / 16.0f, 1.0f / 256.0f);
}

// One 64-group of the lane's rows: row j = 2 * bi + half is row
// lane + 32 * half of row block bi; words of 32-groups 2g and 2g + 1.
template <int RB>
struct Unit {
    uint4 w[2 * RB][2];
    uint32_t m[2 * RB];   // metadata of each row
};

template <int RB>
__device__ __forceinline__ void load_unit(Unit<RB>& u, const uint4* plane_rb,
                                          const uint32_t* meta_rb, size_t qstride, size_t mstride,
                                          int g, int lane, uint64_t pol) {
#pragma unroll
    for (int bi = 0; bi < RB; ++bi) {
        const uint4* q = plane_rb + bi * qstride + (size_t)(2 * g) * 64 + lane;
        u.w[2 * bi][0] = ld_stream(q, pol);
        u.w[2 * bi + 1][0] = ld_stream(q + 32, pol);
        u.w[2 * bi][1] = ld_stream(q + 64, pol);
        u.w[2 * bi + 1][1] = ld_stream(q + 96, pol);
        const uint32_t* m = meta_rb + bi * mstride + (size_t)g * 64 + lane;
        u.m[2 * bi] = ld_stream(m, pol);
        u.m[2 * bi + 1] = ld_stream(m + 32, pol);
    }
}

// T activation rows (m0 .. m0 + T - 1) against the lane's 2 * RB rows of one
// 64-group; the group's contribution is added to the warp's partials
// (redw: [M][64 * RB]). Each x float4 read from shared memory serves all of
// the lane's rows; each decoded word serves all T activation rows.
template <int T, int RB>
__device__ __forceinline__ void tile(Unit<RB>& u, const float* xs, int xrow, int gl,
                                     const float* xsum, int cap, float* redw, int m0, int lane,
                                     uint32_t mg) {
    constexpr int R = 2 * RB;
    float2 acc[R][T];
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
        for (int i = 0; i < T; ++i) acc[j][i] = make_float2(0.0f, 0.0f);
    // Words are consumed from .x and rotated in place: after the four words
    // of a 32-group the unit is back in its original order.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            const float4* xr0 =
                reinterpret_cast<const float4*>(xs + (size_t)m0 * xrow + gl * 64 + h * 32) + c;
            float4 xa[T], xb[T];
#pragma unroll
            for (int i = 0; i < T; ++i) {
                xa[i] = xr0[(size_t)i * (xrow / 4)];
                xb[i] = xr0[(size_t)i * (xrow / 4) + 4];
            }
#pragma unroll
            for (int j = 0; j < R; ++j) {
                float2 f[4];
                decode(u.w[j][h].x, mg, f);
#pragma unroll
                for (int i = 0; i < T; ++i) {
                    acc[j][i] = __ffma2_rn(f[0], make_float2(xa[i].x, xa[i].y), acc[j][i]);
                    acc[j][i] = __ffma2_rn(f[1], make_float2(xa[i].z, xa[i].w), acc[j][i]);
                    acc[j][i] = __ffma2_rn(f[2], make_float2(xb[i].x, xb[i].y), acc[j][i]);
                    acc[j][i] = __ffma2_rn(f[3], make_float2(xb[i].z, xb[i].w), acc[j][i]);
                }
                const uint4 w = u.w[j][h];
                u.w[j][h] = make_uint4(w.y, w.z, w.w, w.x);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
        // bf16 -> f32: the bf16 bits are the top half of the f32 pattern.
        const float s = __uint_as_float(u.m[j] << 16), b = __uint_as_float(u.m[j] & 0xFFFF0000u);
#pragma unroll
        for (int i = 0; i < T; ++i) {
            const float xm = xsum[(m0 + i) * cap + gl];
            redw[(m0 + i) * 64 * RB + (j >> 1) * 64 + (j & 1) * 32 + lane] +=
                fmaf(s, acc[j][i].x + acc[j][i].y, b * xm);
        }
    }
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ float ld_cluster(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// RB row blocks per CTA (each lane owns 2 * RB rows); PF: prefetch the
// warp's next 64-group while computing the current one; TM: the largest
// activation-row tile.
template <int RB, bool PF, int TM>
__global__ void __launch_bounds__(kThreads, 2) af4_gemv_kernel(const Params p) {
    constexpr int NR = 64 * RB;                          // rows per CTA
    extern __shared__ __align__(16) uint8_t smem[];
    const int M = p.M;
    const int xrow = p.cap * 64;                         // floats per staged x row
    float* xs = reinterpret_cast<float*>(smem);          // [M][cap * 64], scaled
    float* xsum = xs + (size_t)M * xrow;                 // [M][cap]
    float* red = xsum + (size_t)M * p.cap;               // [warps][M][NR]
    float* part = red + (size_t)kWarps * M * NR;         // [M][NR]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rb = blockIdx.x * RB;                      // first row block
    const int g0 = blockIdx.y * p.gpc;                   // first 64-group of the K slice
    const uint32_t mg = p.magic;
    const uint64_t pol = l2_evict_first();
    const size_t qstride = (size_t)p.G32 * 64, mstride = (size_t)p.G64 * 64;
    const uint4* plane_rb = p.plane + (size_t)rb * qstride;
    const uint32_t* meta_rb = p.meta + (size_t)rb * mstride;

    for (int i = threadIdx.x; i < kWarps * M * NR; i += kThreads) red[i] = 0.0f;
    float* redw = red + (size_t)warp * M * NR;
    const bool vec = (reinterpret_cast<uintptr_t>(p.x) & 15) == 0;

    for (int s0 = 0; s0 < p.gpc; s0 += p.cap) {
        const int nsub = min(p.cap, p.gpc - s0);
        const int gb = g0 + s0;                          // first 64-group of the sub-slice
        // The weights do not depend on the preceding kernel: issue the first
        // group's loads before waiting for it.
        Unit<RB> u;
        if (warp < nsub) load_unit(u, plane_rb, meta_rb, qstride, mstride, gb + warp, lane, pol);
        if (s0 == 0) {
            pdl_launch_dependents();
            pdl_wait();
        }
        // Stage x (scaled per element) and the per-group sums of the unscaled
        // x: thread i takes 4 consecutive elements, and the 16 lanes of a
        // half-warp cover one 64-group (len and the stride are multiples of
        // 64 elements), whose sum they reduce by shuffles. Each thread issues
        // up to kXB loads before it uses any.
        const int q4 = nsub * 16;
        const int total = M * q4;
        for (int base = warp * 32; base < total; base += kThreads * kXB) {
            float4 v[kXB];
#pragma unroll
            for (int b = 0; b < kXB; ++b) {
                const int i = base + b * kThreads + lane;
                v[b] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (i < total) {
                    const int m = i / q4, kk = 4 * (i - m * q4);
                    const float* src = p.x + (size_t)m * p.K + (size_t)gb * 64 + kk;
                    v[b] = vec ? *reinterpret_cast<const float4*>(src)
                               : make_float4(src[0], src[1], src[2], src[3]);
                }
            }
#pragma unroll
            for (int b = 0; b < kXB; ++b) {
                const int i = base + b * kThreads + lane;
                float t = (v[b].x + v[b].y) + (v[b].z + v[b].w);
#pragma unroll
                for (int off = 8; off >= 1; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
                if (i < total) {
                    const int m = i / q4, kk = 4 * (i - m * q4);
                    const float4 sc = x_scale(kk & 31);
                    *reinterpret_cast<float4*>(xs + (size_t)m * xrow + kk) =
                        make_float4(v[b].x * sc.x, v[b].y * sc.y, v[b].z * sc.z, v[b].w * sc.w);
                    if ((lane & 15) == 0) xsum[m * p.cap + (kk >> 6)] = t;
                }
            }
        }
        __syncthreads();

        for (int gl = warp; gl < nsub; gl += kWarps) {
            if (!PF && gl != warp)
                load_unit(u, plane_rb, meta_rb, qstride, mstride, gb + gl, lane, pol);
            Unit<RB> nx;
            const bool more = PF && gl + kWarps < nsub;
            if (more) load_unit(nx, plane_rb, meta_rb, qstride, mstride, gb + gl + kWarps, lane, pol);
            int m0 = 0;
            if (TM >= 8)
                for (; m0 + 8 <= M; m0 += 8)
                    tile<8, RB>(u, xs, xrow, gl, xsum, p.cap, redw, m0, lane, mg);
            for (; m0 + 4 <= M; m0 += 4) tile<4, RB>(u, xs, xrow, gl, xsum, p.cap, redw, m0, lane, mg);
            if (M - m0 >= 2) {
                tile<2, RB>(u, xs, xrow, gl, xsum, p.cap, redw, m0, lane, mg);
                m0 += 2;
            }
            if (M - m0 >= 1) tile<1, RB>(u, xs, xrow, gl, xsum, p.cap, redw, m0, lane, mg);
            if (more) u = nx;
        }
        __syncthreads();
    }

    // The warps' partials in warp order; then the K slices in rank order.
    const int n0 = rb * 64;
    for (int i = threadIdx.x; i < M * NR; i += kThreads) {
        float v = red[i];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) v += red[(size_t)w * M * NR + i];
        if (p.KS == 1)
            p.y[(size_t)(i / NR) * p.N + n0 + (i % NR)] = v;
        else
            part[i] = v;
    }
    if (p.KS > 1) {
        cluster_sync();
        const int per = M * NR / p.KS;
        const int i0 = (int)cluster_rank() * per;
        const uint32_t base = smem_addr(part);
        for (int i = i0 + threadIdx.x; i < i0 + per; i += kThreads) {
            float v = ld_cluster(base + 4u * i, 0);
            for (int r = 1; r < p.KS; ++r) v += ld_cluster(base + 4u * i, (uint32_t)r);
            p.y[(size_t)(i / NR) * p.N + n0 + (i % NR)] = v;
        }
        // No CTA leaves while another may still read its shared memory.
        cluster_sync();
    }
}

// Shared memory bytes for M rows, an x sub-slice of cap 64-groups and RB
// row blocks per CTA.
size_t smem_bytes(int M, int cap, int RB) {
    return (size_t)M * cap * 64 * 4 + (size_t)M * cap * 4 + (size_t)kWarps * M * 64 * RB * 4 +
           (size_t)M * 64 * RB * 4;
}

template <int RB, bool PF, int TM>
int launch(const DevCtx& dc, const Params& p, int blocks, size_t smem, cudaStream_t s) {
    auto kern = af4_gemv_kernel<RB, PF, TM>;
    static size_t configured[64] = {0};
    if (smem > 48 * 1024 && dc.device >= 0 && dc.device < 64 && configured[dc.device] < smem) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_fail(e);
        configured[dc.device] = smem;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)blocks, (unsigned)p.KS, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (p.KS > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = (unsigned)p.KS;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (launch_option(QG_OPT_PDL) != 0) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
    return e == cudaSuccess ? QG_OK : cuda_fail(e);
}

// Row blocks per CTA: two (four rows per lane) when the block count is even.
int rows_blocks_per_cta(long long N) { return (N / 64) % 2 == 0 ? 2 : 1; }

}  // namespace

int af4_gemv_launch(const DevCtx& dc, const float* x, const uint32_t* plane, const uint32_t* meta,
                    float* y, long long M, long long N, long long K, cudaStream_t s) {
    // One or two rows of x: the register-resident-x kernel when it takes the
    // shape (for both M or for neither).
    if (M <= 2) {
        const int rc = af4_xreg_launch(dc, x, plane, meta, y, M, N, K, s);
        if (rc != QG_ERR_UNSUPPORTED) return rc;
    }
    Params p{};
    p.x = x;
    p.plane = reinterpret_cast<const uint4*>(plane);
    p.meta = meta;
    p.y = y;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.G32 = (int)(K / 32);
    p.G64 = (int)(K / 64);
    p.magic = 0x4B000000u;
    const int RB = rows_blocks_per_cta(N);
    // K slices, each a whole number of 64-groups: for M <= 8 enough CTAs for
    // about one and a half per SM (measured at N = K = 4096: 14.7 us against
    // 25.4 us with half an SM's worth); for larger M, whose x staging and
    // partials take most of an SM's shared memory, about one CTA per two SMs
    // (55 us against 88 us at M = 32).
    const int blocks = (int)(N / 64) / RB;
    const int target = M <= 8 ? (3 * dc.num_sms) / 2 : dc.num_sms / 2;
    int KS = 1;
    while (KS < kMaxKS && blocks * KS < target && p.G64 % (2 * KS) == 0) KS *= 2;
    p.KS = KS;
    p.gpc = p.G64 / KS;
    // x sub-slice: the whole K slice if it fits, else a multiple of the warp
    // count (so that every warp takes the same groups in the same order).
    const size_t limit = (size_t)dc.max_smem_optin;
    int cap = p.gpc;
    if (smem_bytes(p.M, cap, RB) > limit) {
        cap = kWarps;
        while (cap + kWarps < p.gpc && smem_bytes(p.M, cap + kWarps, RB) <= limit) cap += kWarps;
    }
    if (smem_bytes(p.M, cap, RB) > limit) return QG_ERR_UNSUPPORTED;
    p.cap = cap;
    const size_t smem = smem_bytes(p.M, cap, RB);
    return RB == 2 ? launch<2, false, 4>(dc, p, blocks, smem, s)
                   : launch<1, true, 8>(dc, p, blocks, smem, s);
}

}  // namespace qg
