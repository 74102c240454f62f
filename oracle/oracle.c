/*
 * Plain CPU oracle for quantized GEMV with fused dequantization.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library includes, links
 * or calls this file; only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load it. It shares no code, header or table
 * with the CUDA path.
 *
 * Everything here is written straight from the format definitions, slowly and
 * in the most literal order: each weight is dequantized to f32 exactly as the
 * format defines it, and every dot product is accumulated in f64 (a product
 * of two f32 values is exact in f64). Alongside each reference value the
 * oracle returns bound = sum_k |x_k * w_k|, the scale used by the parity
 * tolerance.
 *
 * Sources (by page and section):
 *  - fused_dual_proj_q4_0.rs (mlx-native 0.9.1), module doc and the
 *    preconditions of dispatch_fused_dual_proj_q4_0: Q4_0 blocks of 32
 *    weights, 18 bytes each (fp16 d then 16 nibble bytes), row-major
 *    [N, K/32]; the dual op equals two single mat-vecs.
 *  - q4_k_gemv_v2.rs (ferrum-kernels 0.7.7), module doc: Q4_K super-blocks of
 *    256 weights in 144 bytes, row-major [N, K/256], K % 256 == 0; the test
 *    there interoperates with the GGUF Q4K type, whose field layout is the
 *    reading taken below.
 *  - qmm_affine.rs (mlx-native 0.21.1), test module: the CPU reference
 *    qmm_affine_t_cpu (w = q*s + b per group along K, f64 accumulation),
 *    pack_b4_to_u32 (code j of a u32 word sits at bits 4j) and
 *    prepare_af4_g64 (the prepared layout with 64-groups and bf16 scale and
 *    bias bits, written out below as orc_prepare_af4_g64).
 *  - qkv_split.rs (mlx-native 0.7.1), module doc: per token the fused row is
 *    [Q | K | V]; every element goes to exactly one output.
 *
 * Readings where the pages are silent (the kernels themselves are not on the
 * pages):
 *  - Q4_0 nibble order: byte 2+j of a block holds element j in its low
 *    nibble and element 16+j in its high nibble; w = (q - 8) * d.
 *  - Q4_K: bytes 0-1 d, 2-3 dmin (fp16, little-endian), 4-15 twelve bytes of
 *    packed 6-bit (scale, min) pairs for 8 sub-blocks of 32, 16-143 nibbles;
 *    w = (d*sc)*q - dmin*m, one f32 rounding (both products are exact).
 *  - Affine: the dequantized weight is fmaf(q, s, b), one f32 rounding; the
 *    packed form holds element 2i in the low nibble of byte i.
 *
 * Parity pins for every function live in tests/test_oracle_*.py. The
 * ORACLE_PLANT_* macros exist only so that a test can build a deliberately
 * wrong copy of this file and check that the pins catch it; the normal build
 * defines none of them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary16 -> binary32, decoded from the bit fields.               */
/* sign (1) | exponent (5, bias 15) | mantissa (10).                          */
/* Every finite half is exactly representable in float, so building the    */
/* value in double and narrowing is exact.                                   */
/* ------------------------------------------------------------------------ */
ORC_API float orc_half_to_float(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1F;
    const int mant = h & 0x3FF;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)mant, -24); /* zero or subnormal: mant * 2^-24 */
    } else if (expo == 31) {
        if (mant != 0) return sign ? -NAN : NAN;
        mag = INFINITY;
    } else {
        mag = ldexp((double)(1024 + mant), expo - 25); /* (1.mant) * 2^(e-15) */
    }
    return (float)(sign ? -mag : mag);
}

static uint16_t rd_u16le(const uint8_t* p) {
    return (uint16_t)(p[0] | ((uint16_t)p[1] << 8));
}

/* ------------------------------------------------------------------------ */
/* Q4_0                                                                      */
/* ------------------------------------------------------------------------ */
#define Q4_0_QK 32
#define Q4_0_BLOCK_BYTES 18

/* Dequantize one Q4_0 block (18 bytes) into 32 floats. */
ORC_API void orc_q4_0_block(const uint8_t* blk, float* out32) {
    const float d = orc_half_to_float(rd_u16le(blk));
    for (int j = 0; j < 16; ++j) {
        const uint8_t byte = blk[2 + j];
#ifdef ORACLE_PLANT_NIBBLE_SWAP
        const int q_lo = byte >> 4, q_hi = byte & 0x0F;
#else
        const int q_lo = byte & 0x0F;
        const int q_hi = byte >> 4;
#endif
#ifdef ORACLE_PLANT_DROP_OFFSET
        out32[j] = (float)q_lo * d;
        out32[16 + j] = (float)q_hi * d;
#else
        out32[j] = (float)(q_lo - 8) * d;      /* exact: 4-bit int x 11-bit d */
        out32[16 + j] = (float)(q_hi - 8) * d;
#endif
    }
}

/* Dequantize rows [0, N) of a Q4_0 matrix into out[N, K]. */
ORC_API void orc_dequant_q4_0(const uint8_t* w, int64_t N, int64_t K, float* out) {
    const int64_t nb = K / Q4_0_QK;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b)
            orc_q4_0_block(w + (n * nb + b) * Q4_0_BLOCK_BYTES, out + n * K + b * Q4_0_QK);
}

/* ------------------------------------------------------------------------ */
/* Q4_K                                                                      */
/* ------------------------------------------------------------------------ */
#define Q4_K_QK 256
#define Q4_K_BLOCK_BYTES 144

/* The 6-bit (scale, min) pair of sub-block j from the 12 packed bytes.
 * j < 4 : low 6 bits of bytes j and j+4.
 * j >= 4: low 4 bits from the two nibbles of byte j+4, top 2 bits from the
 *         top 2 bits of bytes j-4 (scale) and j (min). */
ORC_API void orc_q4_k_scale_min(const uint8_t* s12, int j, int* sc, int* m) {
    if (j < 4) {
        *sc = s12[j] & 63;
        *m = s12[j + 4] & 63;
    } else {
#ifdef ORACLE_PLANT_Q4K_HIGH_BITS
        *sc = (s12[j + 4] & 0x0F) | ((s12[j] >> 6) << 4);
        *m = (s12[j + 4] >> 4) | ((s12[j - 4] >> 6) << 4);
#else
        *sc = (s12[j + 4] & 0x0F) | ((s12[j - 4] >> 6) << 4);
        *m = (s12[j + 4] >> 4) | ((s12[j] >> 6) << 4);
#endif
    }
}

/* Dequantize one 144-byte super-block into 256 floats. Nibble chunk c (32
 * bytes) holds sub-block 2c in its low nibbles and 2c+1 in its high ones. */
ORC_API void orc_q4_k_block(const uint8_t* blk, float* out256) {
    const float d = orc_half_to_float(rd_u16le(blk));
    const float dmin = orc_half_to_float(rd_u16le(blk + 2));
    const uint8_t* s12 = blk + 4;
    const uint8_t* qs = blk + 16;
    for (int c = 0; c < 4; ++c) {
        int sc0, m0, sc1, m1;
        orc_q4_k_scale_min(s12, 2 * c, &sc0, &m0);
        orc_q4_k_scale_min(s12, 2 * c + 1, &sc1, &m1);
        const float ds0 = d * (float)sc0, dm0 = dmin * (float)m0; /* exact */
        const float ds1 = d * (float)sc1, dm1 = dmin * (float)m1; /* exact */
        for (int l = 0; l < 32; ++l) {
            const uint8_t byte = qs[32 * c + l];
            const float p0 = ds0 * (float)(byte & 0x0F); /* exact */
            const float p1 = ds1 * (float)(byte >> 4);   /* exact */
            out256[64 * c + l] = p0 - dm0;               /* one rounding */
            out256[64 * c + 32 + l] = p1 - dm1;
        }
    }
}

ORC_API void orc_dequant_q4_k(const uint8_t* w, int64_t N, int64_t K, float* out) {
    const int64_t nb = K / Q4_K_QK;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b)
            orc_q4_k_block(w + (n * nb + b) * Q4_K_BLOCK_BYTES, out + n * K + b * Q4_K_QK);
}

/* ------------------------------------------------------------------------ */
/* Affine group quantization                                                 */
/* ------------------------------------------------------------------------ */
/* Code of element (n, k): one byte each, or two per byte (low nibble = even
 * k), the byte view of a u32 word whose code j sits at bits 4j. */
static int affine_code(const uint8_t* q, int64_t n, int64_t k, int64_t K, int packed) {
    if (packed) {
        const uint8_t byte = q[n * (K / 2) + k / 2];
        return (k & 1) ? (byte >> 4) : (byte & 0x0F);
    }
    return q[n * K + k];
}

ORC_API void orc_dequant_affine_row(const uint8_t* q, const float* s, const float* b, int64_t n,
                                    int64_t K, int gs, int packed, float* out_row) {
    const int64_t G = K / gs;
    for (int64_t k = 0; k < K; ++k) {
        const float code = (float)affine_code(q, n, k, K, packed);
        out_row[k] = fmaf(code, s[n * G + k / gs], b[n * G + k / gs]);
    }
}

ORC_API void orc_dequant_affine(const uint8_t* q, const float* s, const float* b, int64_t N,
                                int64_t K, int gs, int packed, float* out) {
    for (int64_t n = 0; n < N; ++n) orc_dequant_affine_row(q, s, b, n, K, gs, packed, out + n * K);
}

/* ------------------------------------------------------------------------ */
/* y[m, n] = sum_k x[m, k] * w[n, k], accumulated in f64.                    */
/* ------------------------------------------------------------------------ */
/* Dot of one dequantized row with every input row: ref[m*N+n], bound[m*N+n]. */
static void dot_row(const float* wrow, const float* x, int64_t M, int64_t N, int64_t K, int64_t n,
                    double* ref, double* bound) {
    for (int64_t m = 0; m < M; ++m) {
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; ++k) {
#ifdef ORACLE_PLANT_X_INDEX
            const double t = (double)x[m * K + (K - 1 - k)] * (double)wrow[k];
#else
            const double t = (double)x[m * K + k] * (double)wrow[k]; /* exact in f64 */
#endif
            acc += t;
            mag += fabs(t);
        }
        ref[m * N + n] = acc;
        if (bound) bound[m * N + n] = mag;
    }
}

/* Dense reference on an already dequantized W[N, K]. */
ORC_API void orc_gemv_dense(const float* W, const float* x, int64_t M, int64_t N, int64_t K,
                            double* ref, double* bound) {
    for (int64_t n = 0; n < N; ++n) dot_row(W + n * K, x, M, N, K, n, ref, bound);
}

/* Quantized references. `rows` lists the output columns n to compute (all
 * of them when rows == NULL); entries of ref/bound for other n are left
 * untouched. Each listed row is dequantized with the functions above, then
 * dotted in f64. */
ORC_API int orc_gemv_q4_0(const uint8_t* w, const float* x, int64_t M, int64_t N, int64_t K,
                          const int64_t* rows, int64_t nrows, double* ref, double* bound) {
    float* wrow = (float*)malloc(sizeof(float) * (size_t)K);
    if (!wrow) return -1;
    const int64_t cnt = rows ? nrows : N;
    for (int64_t i = 0; i < cnt; ++i) {
        const int64_t n = rows ? rows[i] : i;
        orc_dequant_q4_0(w + n * (K / Q4_0_QK) * Q4_0_BLOCK_BYTES, 1, K, wrow);
        dot_row(wrow, x, M, N, K, n, ref, bound);
    }
    free(wrow);
    return 0;
}

ORC_API int orc_gemv_q4_k(const uint8_t* w, const float* x, int64_t M, int64_t N, int64_t K,
                          const int64_t* rows, int64_t nrows, double* ref, double* bound) {
    float* wrow = (float*)malloc(sizeof(float) * (size_t)K);
    if (!wrow) return -1;
    const int64_t cnt = rows ? nrows : N;
    for (int64_t i = 0; i < cnt; ++i) {
        const int64_t n = rows ? rows[i] : i;
        orc_dequant_q4_k(w + n * (K / Q4_K_QK) * Q4_K_BLOCK_BYTES, 1, K, wrow);
        dot_row(wrow, x, M, N, K, n, ref, bound);
    }
    free(wrow);
    return 0;
}

ORC_API int orc_qmm_affine(const float* x, const uint8_t* q, const float* s, const float* b,
                           int64_t M, int64_t N, int64_t K, int gs, int packed,
                           const int64_t* rows, int64_t nrows, double* ref, double* bound) {
    float* wrow = (float*)malloc(sizeof(float) * (size_t)K);
    if (!wrow) return -1;
    const int64_t cnt = rows ? nrows : N;
    for (int64_t i = 0; i < cnt; ++i) {
        const int64_t n = rows ? rows[i] : i;
        orc_dequant_affine_row(q, s, b, n, K, gs, packed, wrow);
        dot_row(wrow, x, M, N, K, n, ref, bound);
    }
    free(wrow);
    return 0;
}

/* The fused dual projection is, by its stated contract, two independent
 * single projections sharing x. */
ORC_API int orc_gemv_dual_q4_0(const uint8_t* w_a, const uint8_t* w_b, const float* x, int64_t M,
                               int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                               double* ref_a, double* bound_a, double* ref_b, double* bound_b) {
    int rc = orc_gemv_q4_0(w_a, x, M, N, K, rows, nrows, ref_a, bound_a);
    if (rc) return rc;
    return orc_gemv_q4_0(w_b, x, M, N, K, rows, nrows, ref_b, bound_b);
}

/* ------------------------------------------------------------------------ */
/* QKV split: qkv[t, :] = [Q (q_sp) | K (k_sp) | V (v_sp)], copied as 32-bit  */
/* words so that every bit pattern (NaN payloads included) survives.         */
/* ------------------------------------------------------------------------ */
ORC_API void orc_qkv_split(const uint32_t* qkv, uint32_t* q, uint32_t* k, uint32_t* v, int64_t seq,
                           int64_t q_sp, int64_t k_sp, int64_t v_sp) {
    const int64_t ch = q_sp + k_sp + v_sp;
    for (int64_t t = 0; t < seq; ++t) {
        const uint32_t* row = qkv + t * ch;
        for (int64_t j = 0; j < q_sp; ++j) q[t * q_sp + j] = row[j];
        for (int64_t j = 0; j < k_sp; ++j) k[t * k_sp + j] = row[q_sp + j];
        for (int64_t j = 0; j < v_sp; ++j) v[t * v_sp + j] = row[q_sp + k_sp + j];
    }
}

/* ------------------------------------------------------------------------ */
/* The prepared AF4-g64 layout. Page: qmm_affine.rs (mlx-native 0.21.1),     */
/* prepare_af4_g64 in the test module, written out here as the definition:  */
/*   plane[((r / 64) * K/32 + g) * 64 + r % 64][c] (g: 32-wide group, c: 0..3)*/
/*   holds, for each pair p = 0..3 with e = 32 g + 16 (p / 2) + 4 c + 2 (p % 2),*/
/*   code[r][e] in bits 4p.. and code[r][e + 1] in bits 16 + 4p..;           */
/*   meta[((r / 64) * K/64 + h) * 64 + r % 64] = scale bits | bias bits << 16 */
/*   for the 64-wide group h.                                                */
/* Parity pins: a hand-computed word (tests/golden/af4_g64.json) and the     */
/* round trip through orc_af4_unpack.                                        */
/* ------------------------------------------------------------------------ */
ORC_API void orc_prepare_af4_g64(const uint8_t* codes, const uint16_t* scales,
                                 const uint16_t* biases, int64_t N, int64_t K, uint32_t* plane,
                                 uint32_t* meta) {
    const int64_t g32n = K / 32, g64n = K / 64;
    for (int64_t r = 0; r < N; ++r) {
        for (int64_t h = 0; h < g64n; ++h)
            meta[((r / 64) * g64n + h) * 64 + r % 64] =
                (uint32_t)scales[r * g64n + h] | ((uint32_t)biases[r * g64n + h] << 16);
        for (int64_t g = 0; g < g32n; ++g)
            for (int c = 0; c < 4; ++c) {
                uint32_t word = 0;
                for (int p = 0; p < 4; ++p) {
                    const int64_t e = g * 32 + 16 * (p / 2) + 4 * c + 2 * (p % 2);
#ifdef ORACLE_PLANT_AF4_HALVES
                    word |= (uint32_t)(codes[r * K + e + 1] & 15u) << (4 * p);
                    word |= (uint32_t)(codes[r * K + e] & 15u) << (16 + 4 * p);
#else
                    word |= (uint32_t)(codes[r * K + e] & 15u) << (4 * p);
                    word |= (uint32_t)(codes[r * K + e + 1] & 15u) << (16 + 4 * p);
#endif
                }
#ifdef ORACLE_PLANT_AF4_ROW_MAJOR
                plane[(r * g32n + g) * 4 + c] = word;
#else
                plane[(((r / 64) * g32n + g) * 64 + r % 64) * 4 + c] = word;
#endif
            }
    }
}

/* The inverse: codes [N, K] and the bf16 bits back from plane and meta. */
ORC_API void orc_af4_unpack(const uint32_t* plane, const uint32_t* meta, int64_t N, int64_t K,
                            uint8_t* codes, uint16_t* scales, uint16_t* biases) {
    const int64_t g32n = K / 32, g64n = K / 64;
    for (int64_t r = 0; r < N; ++r) {
        for (int64_t h = 0; h < g64n; ++h) {
            const uint32_t m = meta[((r / 64) * g64n + h) * 64 + r % 64];
            scales[r * g64n + h] = (uint16_t)(m & 0xFFFFu);
            biases[r * g64n + h] = (uint16_t)(m >> 16);
        }
        for (int64_t g = 0; g < g32n; ++g)
            for (int c = 0; c < 4; ++c) {
                const uint32_t word = plane[(((r / 64) * g32n + g) * 64 + r % 64) * 4 + c];
                for (int p = 0; p < 4; ++p) {
                    const int64_t e = g * 32 + 16 * (p / 2) + 4 * c + 2 * (p % 2);
                    codes[r * K + e] = (uint8_t)((word >> (4 * p)) & 15u);
                    codes[r * K + e + 1] = (uint8_t)((word >> (16 + 4 * p)) & 15u);
                }
            }
    }
}

/* bfloat16 bits -> float: the top 16 bits of the f32 pattern. */
ORC_API float orc_bf16_to_float(uint16_t h) {
    const uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}
