/*
 * mxq_oracle.c -- plain, slow, obviously correct CPU oracle for the MXFP8
 * grouped-quantization + grouped-GEMM hot path of an MoE expert layer.
 *
 * TEST INFRASTRUCTURE ONLY. This file is compiled into its own shared
 * library and is loaded only by the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg. It shares no source, header, table or
 * helper with the CUDA path and must never be reached from it.
 *
 * Sources of the definitions (cited per function below):
 *   [RQ]  TransformerEngine PR #3244, "[Pytorch] Add support for row-wise
 *         quanted input for grouped gemm": description, the review threads on
 *         prepare_prequantized_mxfp8_grouped_input (compact scale shape, the
 *         128-token per-expert alignment, swizzle of the dispatch scales,
 *         group_dequantize then columnwise group_quantize) and the Greptile
 *         flowchart (dequantize -> columnwise requantize -> wgrad; bias
 *         reductions from the dequantized tensor).
 *   [FM]  TransformerEngine PR #3545, "Fix distributed BF16 weights and trim
 *         NVFP4 saved state in the fused grouped MLP": description and commit
 *         notes (forward GEMMs read rowwise weights, dgrad the columnwise
 *         weight copy, wgrad only columnwise input tiles; FC1 -> activation ->
 *         FC2 fused grouped MLP).
 *   [DI]  TransformerEngine PR #3224, "Improve device-init grouped linear
 *         module with single grouped weight support": Greptile summary
 *         (device m_splits, single grouped weight (E,out,in) and 2-D grouped
 *         bias, per-member swizzled scale bases in group_quantize_mxfp8).
 *   [MX]  OCP Microscaling Formats (MX) v1.0: E4M3 element format (bias 7,
 *         max finite 448, no infinities), E8M0 shared scale, shared exponent
 *         floor(log2(amax)) - emax_elem with emax_elem(E4M3) = 8.
 *   [SW]  The 128x4 tensor-core block-scale layout published in the PTX ISA
 *         (tcgen05 block-scaling, scale-factor layout) and the cuBLAS
 *         block-scaling documentation.
 *
 * Readings taken where the pages are silent (each repeated at its function):
 *   - element cast: round to nearest, ties to even, saturating at +-448,
 *     sign kept (negative values that round to zero give -0 = 0x80);
 *   - all-zero block: scale code 0x00 (2^-127); exponent clamped to
 *     [-127, 127];
 *   - colwise compact scale shape is the transpose of the page's rowwise
 *     rule: (round_up(M/32,4), round_up(K,128)), zero padded;
 *   - colwise E4M3 bytes keep the (M,K) byte order of the source;
 *   - dequantization is exact (the page's bf16 dequant is exact for every
 *     value these workloads produce);
 *   - SwiGLU takes the first half of the FC1 output as the gate.
 *
 * Floating point: everything is computed in double; scaling by powers of two
 * uses ldexp (exact) and rounding uses nearbyint under the default
 * round-to-nearest-even mode.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------ codecs */

/* bf16 bit pattern -> exact value (bf16 is the top half of an IEEE binary32). */
ORC_API double orc_bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), with one rounding.
 * bf16: 8 significant bits, exponents -126..127, subnormal quantum 2^-133. */
ORC_API uint16_t orc_bf16_round(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7F80;
    int e;
    frexp(a, &e);
    int E = e - 1;                 /* floor(log2 a) */
    if (E < -126) E = -126;        /* subnormal range shares the last quantum */
    double quantum = ldexp(1.0, E - 7);
    double r = nearbyint(a / quantum) * quantum;
    if (r >= ldexp(1.0, 128)) return sign | 0x7F80;
    float f = (float)r;            /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return sign | (uint16_t)(u >> 16);
}

/* E4M3 code -> value [MX]: S.EEEE.MMM, bias 7, subnormals m*2^-9,
 * 0x7F/0xFF are NaN (never produced by the encoder). */
ORC_API double orc_e4m3_value(uint8_t c) {
    int s = c >> 7, E = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (E == 0xF && m == 7) return NAN;
    if (E == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, E - 7);
    return s ? -v : v;
}

/* value -> E4M3 code [MX], round to nearest even, saturating finite.
 * Reading: the sign is kept, so negatives that round to zero give 0x80. */
ORC_API uint8_t orc_e4m3_encode(double v) {
    uint8_t sign = signbit(v) ? 0x80 : 0;
    double a = fabs(v);
    if (isnan(v)) return sign | 0x7F;           /* out of contract */
    if (a > 448.0) return sign | 0x7E;          /* saturate to max finite */
    if (a < ldexp(1.0, -6)) {                   /* subnormal: step 2^-9 */
        double q = nearbyint(ldexp(a, 9));      /* 0..8; 8 is the code of 2^-6 */
        return sign | (uint8_t)q;
    }
    int e;
    frexp(a, &e);
    int E = e - 1;                              /* -6..8 */
    double frac = ldexp(a, -E) - 1.0;           /* [0,1) exactly */
    double q = nearbyint(frac * 8.0);           /* 0..8 */
    if (q == 8.0) { q = 0.0; E += 1; }
    return sign | (uint8_t)(((E + 7) << 3) | (int)q);
}

/* Shared exponent of a block [MX]: s = floor(log2 amax) - 8, clamped to
 * [-127, 127]; an all-zero block gives s = -127 (reading). The E8M0 code is
 * s + 127; code 0xFF (NaN) is never produced. */
ORC_API int orc_e8m0_exponent(double amax) {
    if (amax == 0.0) return -127;
    int e;
    frexp(amax, &e);
    int s = (e - 1) - 8;
    if (s < -127) s = -127;
    if (s > 127) s = 127;
    return s;
}

ORC_API double orc_e8m0_value(uint8_t code) { return ldexp(1.0, (int)code - 127); }

/* Element-wise loops over the scalar definitions above (for exhaustive tests). */
ORC_API void orc_e4m3_encode_n(const double* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}
ORC_API void orc_e8m0_exponent_n(const double* a, int64_t n, int32_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e8m0_exponent(a[i]);
}
ORC_API void orc_bf16_round_n(const double* v, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_round(v[i]);
}

/* One MX block [MX] [RQ]: amax, shared exponent, elements cast after
 * scaling by 2^-s. n is 32 for every call in this file. */
ORC_API void orc_quantize_block(const double* v, int n, uint8_t* codes, uint8_t* scale_code) {
    double amax = 0.0;
    for (int i = 0; i < n; ++i) amax = fmax(amax, fabs(v[i]));
    int s = orc_e8m0_exponent(amax);
    *scale_code = (uint8_t)(s + 127);
    for (int i = 0; i < n; ++i) codes[i] = orc_e4m3_encode(ldexp(v[i], -s));
}

/* ----------------------------------------------------------------- layouts */

static int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

/* Byte offset of logical scale S[r][c] (R x C, R%128 == 0, C%4 == 0) in the
 * 128x4 tensor-core scale layout [SW]: 512-byte atoms of 128 rows x 4 cols,
 * atoms row-major over (R/128, C/4); inside an atom row r%32 owns 16 bytes
 * holding rows r%32 + 32*j (j = 0..3) x 4 columns. */
ORC_API int64_t orc_swizzle_offset(int64_t r, int64_t c, int64_t C) {
    return ((r / 128) * (C / 4) + c / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

/* Scatter a logical R x C scale matrix (element (r,c) at S[r*sr + c*sc]) into
 * the swizzled layout at out. */
ORC_API void orc_swizzle(const uint8_t* S, int64_t R, int64_t C, int64_t sr, int64_t sc, uint8_t* out) {
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) out[orc_swizzle_offset(r, c, C)] = S[r * sr + c * sc];
}

/* Compact (unswizzled) scale shapes [RQ]: rowwise (round_up(M,128),
 * round_up(K/32,4)); colwise (reading, the transpose of the rowwise rule)
 * (round_up(M/32,4), round_up(K,128)). Pad bytes are zero. */
ORC_API void orc_compact_shape(int64_t M, int64_t K, int colwise, int64_t* rows, int64_t* cols) {
    if (!colwise) { *rows = round_up(M, 128); *cols = round_up(K / 32, 4); }
    else          { *rows = round_up(M / 32, 4); *cols = round_up(K, 128); }
}

/* --------------------------------------------------------------- quantize */

/* Rowwise MX quantization [RQ] of an M x K matrix given as doubles: blocks
 * are x[m, 32j:32j+32]. Scales go to the compact layout (ld = ldS). */
static void quantize_rowwise_f64(const double* x, int64_t M, int64_t K, uint8_t* q, uint8_t* S, int64_t ldS) {
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < K / 32; ++j)
            orc_quantize_block(x + m * K + 32 * j, 32, q + m * K + 32 * j, S + m * ldS + j);
}

/* Colwise MX quantization [RQ]: blocks are x[32i:32i+32, k] (along tokens).
 * Codes keep the (M,K) byte order (reading); scales compact (ld = ldS). */
static void quantize_colwise_f64(const double* x, int64_t M, int64_t K, uint8_t* q, uint8_t* S, int64_t ldS) {
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M / 32; ++i) {
        double v[32];
        uint8_t c[32];
        for (int64_t k = 0; k < K; ++k) {
            for (int t = 0; t < 32; ++t) v[t] = x[(32 * i + t) * K + k];
            orc_quantize_block(v, 32, c, S + i * ldS + k);
            for (int t = 0; t < 32; ++t) q[(32 * i + t) * K + k] = c[t];
        }
    }
}

static double* bf16_matrix_to_f64(const uint16_t* x, int64_t n) {
    double* d = (double*)malloc((size_t)n * sizeof(double));
    if (!d) return NULL;
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) d[i] = orc_bf16_value(x[i]);
    return d;
}

/* Check the grouping contract [RQ] [DI]: m_e >= 0, m_e % 128 == 0 (the
 * dispatch's per-expert alignment), sum == M. Returns 0 when valid. */
ORC_API int orc_check_splits(const int64_t* m_splits, int E, int64_t M) {
    int64_t sum = 0;
    for (int e = 0; e < E; ++e) {
        if (m_splits[e] < 0 || m_splits[e] % 128) return -1;
        sum += m_splits[e];
    }
    return sum == M ? 0 : -1;
}

/* Grouped MXFP8 quantization of a token-major bf16 X (M x K) split into E
 * experts by m_splits [RQ] [DI]. With every m_e a multiple of 128 no 32-block
 * straddles two experts, so rowwise and colwise blocks are those of the whole
 * matrix; the grouping only decides the colwise swizzled scale bases.
 *
 * Outputs (NULL to skip): row_q (M,K) + row_s, col_q (M,K) + col_s.
 * swizzled == 0: compact scales (shapes of orc_compact_shape, zero padded).
 * swizzled != 0: row_s is the swizzle of the (M, K/32) rowwise scales as one
 * matrix; col_s holds, for each expert e, the swizzle of the logical
 * (K, m_e/32) matrix S_e[k][i] = scale of token block i of expert e at column
 * k, placed at byte K*off_e/32 ("per-member swizzled scale bases" [DI]). */
ORC_API int orc_group_quantize(const uint16_t* x, int64_t M, int64_t K, int E, const int64_t* m_splits,
                               int swizzled, uint8_t* row_q, uint8_t* row_s, uint8_t* col_q, uint8_t* col_s) {
    if (K % 128 || orc_check_splits(m_splits, E, M)) return -1;
    double* d = bf16_matrix_to_f64(x, M * K);
    if (!d) return -2;
    int64_t rr, rc, cr, cc;
    orc_compact_shape(M, K, 0, &rr, &rc);
    orc_compact_shape(M, K, 1, &cr, &cc);
    if (row_q) {
        uint8_t* S = (uint8_t*)calloc((size_t)(rr * rc), 1);
        quantize_rowwise_f64(d, M, K, row_q, S, rc);
        if (!swizzled) memcpy(row_s, S, (size_t)(rr * rc));
        else orc_swizzle(S, M, K / 32, rc, 1, row_s);
        free(S);
    }
    if (col_q) {
        uint8_t* S = (uint8_t*)calloc((size_t)(cr * cc), 1);
        quantize_colwise_f64(d, M, K, col_q, S, cc);
        if (!swizzled) memcpy(col_s, S, (size_t)(cr * cc));
        else {
            int64_t off = 0;
            for (int e = 0; e < E; ++e) {
                int64_t me = m_splits[e];
                if (me) orc_swizzle(S + (off / 32) * cc, K, me / 32, 1, cc, col_s + K * off / 32);
                off += me;
            }
        }
        free(S);
    }
    free(d);
    return 0;
}

/* -------------------------------------------------------------- dequantize */

/* Rowwise dequantization [RQ] (group_dequantize needs compact scales):
 * deq[m,k] = e4m3(q[m,k]) * 2^(s[m, k/32] - 127), exact. */
ORC_API void orc_dequant_rowwise(const uint8_t* q, const uint8_t* S_compact, int64_t M, int64_t K, double* out) {
    int64_t rr, rc;
    orc_compact_shape(M, K, 0, &rr, &rc);
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            out[m * K + k] = ldexp(orc_e4m3_value(q[m * K + k]), (int)S_compact[m * rc + k / 32] - 127);
}

/* Colwise dequantization: deq[m,k] = e4m3(q[m,k]) * 2^(s[m/32, k] - 127). */
ORC_API void orc_dequant_colwise(const uint8_t* q, const uint8_t* S_compact, int64_t M, int64_t K, double* out) {
    int64_t cr, cc;
    orc_compact_shape(M, K, 1, &cr, &cc);
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            out[m * K + k] = ldexp(orc_e4m3_value(q[m * K + k]), (int)S_compact[(m / 32) * cc + k] - 127);
}

/* ----------------------------------------------------------------- requant */

/* Columnwise copy of a rowwise-prequantized grouped input [RQ] (the
 * expert-parallel FP8 dispatch delivers rowwise data with compact scales):
 *   1. dequantize the rowwise data with its compact scales;
 *   2. quantize the dequantized values columnwise (a double quantization;
 *      it is NOT the colwise quantization of any original source);
 *   3. emit the rowwise scales in the GEMM (swizzled) layout for fprop/dgrad;
 *   4. optionally reduce dbias per expert from the dequantized values and
 *      write the dequantized tensor as bf16.
 * col_s layout follows `swizzled` as in orc_group_quantize. dbias (E,K) is
 * the fp64 sum over each expert's rows (0 for an empty expert). */
ORC_API int orc_requant_colwise(const uint8_t* row_q, const uint8_t* row_s_compact, int64_t M, int64_t K, int E,
                                const int64_t* m_splits, int swizzled, uint8_t* col_q, uint8_t* col_s,
                                uint8_t* row_s_swizzled, double* dbias, uint16_t* deq_bf16) {
    if (K % 128 || orc_check_splits(m_splits, E, M)) return -1;
    double* d = (double*)malloc((size_t)(M * K) * sizeof(double));
    if (!d) return -2;
    orc_dequant_rowwise(row_q, row_s_compact, M, K, d);
    int64_t rr, rc, cr, cc;
    orc_compact_shape(M, K, 0, &rr, &rc);
    orc_compact_shape(M, K, 1, &cr, &cc);
    if (col_q) {
        uint8_t* S = (uint8_t*)calloc((size_t)(cr * cc), 1);
        quantize_colwise_f64(d, M, K, col_q, S, cc);
        if (!swizzled) memcpy(col_s, S, (size_t)(cr * cc));
        else {
            int64_t off = 0;
            for (int e = 0; e < E; ++e) {
                int64_t me = m_splits[e];
                if (me) orc_swizzle(S + (off / 32) * cc, K, me / 32, 1, cc, col_s + K * off / 32);
                off += me;
            }
        }
        free(S);
    }
    if (row_s_swizzled) orc_swizzle(row_s_compact, M, K / 32, rc, 1, row_s_swizzled);
    if (dbias) {
        int64_t off = 0;
        for (int e = 0; e < E; ++e) {
            #pragma omp parallel for schedule(static)
            for (int64_t k = 0; k < K; ++k) {
                double acc = 0.0;
                for (int64_t m = off; m < off + m_splits[e]; ++m) acc += d[m * K + k];
                dbias[e * K + k] = acc;
            }
            off += m_splits[e];
        }
    }
    if (deq_bf16) {
        #pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < M * K; ++i) deq_bf16[i] = orc_bf16_round(d[i]);
    }
    free(d);
    return 0;
}

/* ------------------------------------------------------------------- dbias */

/* Per-expert bias gradient [RQ]: db[e,n] = sum over expert e's rows of
 * dY[m,n], in fp64; an empty expert gives 0. */
ORC_API int orc_grouped_dbias(const uint16_t* dy, int64_t M, int64_t N, int E, const int64_t* m_splits, double* out) {
    if (orc_check_splits(m_splits, E, M)) return -1;
    int64_t off = 0;
    for (int e = 0; e < E; ++e) {
        #pragma omp parallel for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t m = off; m < off + m_splits[e]; ++m) acc += orc_bf16_value(dy[m * N + n]);
            out[e * N + n] = acc;
        }
        off += m_splits[e];
    }
    return 0;
}

/* Scaled bias and routing-scale gradients [RQ: bias and routing-scale
 * reductions are taken from the dequantized gradient]. Reading (the pages do
 * not print the formula): expert e adds its bias scaled by the token's
 * routing scale, y[m,:] = X[m,:] W_e^T + s_m * b_e, so for the gradient dY
 *   db[e,n] = sum over expert e's rows m of s_m * dY[m,n]
 *   ds[m]   = sum over n of dY[m,n] * b_e(m)[n]
 * in fp64. dy holds the exact values (bf16 widened, or the dequantized
 * rowwise wire format); bias is bf16 bits (E, N); probs fp32 (M). Either
 * output may be NULL. An empty expert gives db = 0. */
ORC_API int orc_scaled_bias_grads(const double* dy, int64_t M, int64_t N, int E, const int64_t* m_splits,
                                  const float* probs, const uint16_t* bias, double* dbias, double* dprobs) {
    if (orc_check_splits(m_splits, E, M)) return -1;
    int64_t off = 0;
    for (int e = 0; e < E; ++e) {
        const int64_t end = off + m_splits[e];
        if (dbias) {
            #pragma omp parallel for schedule(static)
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t m = off; m < end; ++m) acc += (double)probs[m] * dy[m * N + n];
                dbias[e * N + n] = acc;
            }
        }
        if (dprobs) {
            #pragma omp parallel for schedule(static)
            for (int64_t m = off; m < end; ++m) {
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) acc += dy[m * N + n] * orc_bf16_value(bias[e * N + n]);
                dprobs[m] = acc;
            }
        }
        off = end;
    }
    return 0;
}

/* ------------------------------------------------------------------- GEMMs */

/* Each GEMM entry is the textbook dot product of dequantized operands in
 * fp64, together with the dot product of their magnitudes (the scale of the
 * rounding error an fp32 accumulation may make). Operands are given by their
 * E4M3 bytes and COMPACT scales; which quantized copy each GEMM reads follows
 * [RQ] [FM]: fprop and dgrad read rowwise activations/gradients, dgrad the
 * columnwise weight copy, wgrad only columnwise copies. */

static inline double deq_row(const uint8_t* q, const uint8_t* S, int64_t ldS, int64_t K, int64_t m, int64_t k) {
    return ldexp(orc_e4m3_value(q[m * K + k]), (int)S[m * ldS + k / 32] - 127);
}
static inline double deq_col(const uint8_t* q, const uint8_t* S, int64_t ldS, int64_t K, int64_t m, int64_t k) {
    return ldexp(orc_e4m3_value(q[m * K + k]), (int)S[(m / 32) * ldS + k] - 127);
}

static int expert_of_row(const int64_t* m_splits, int E, int64_t m, int64_t* off_out) {
    int64_t off = 0;
    for (int e = 0; e < E; ++e) {
        if (m < off + m_splits[e]) { if (off_out) *off_out = off; return e; }
        off += m_splits[e];
    }
    return -1;
}

/* fprop [RQ] [DI]: Y[m,n] = sum_k X[m,k] * W[e(m),n,k] (+ b[e(m),n]).
 * X rowwise (M,K), W rowwise (E*N, K) with compact scales, bias bf16 (E,N)
 * or NULL. Evaluates the entries listed in (rows[i], cols[i]). */
ORC_API void orc_fprop_entries(const uint8_t* xq, const uint8_t* xs, const uint8_t* wq, const uint8_t* ws,
                               const uint16_t* bias, int64_t M, int64_t N, int64_t K, int E, const int64_t* m_splits,
                               int64_t count, const int64_t* rows, const int64_t* cols, double* val, double* mag) {
    int64_t xr, xc, wr, wc;
    orc_compact_shape(M, K, 0, &xr, &xc);
    orc_compact_shape((int64_t)E * N, K, 0, &wr, &wc);
    #pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = rows[i], n = cols[i];
        int e = expert_of_row(m_splits, E, m, NULL);
        double acc = 0.0, am = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = deq_row(xq, xs, xc, K, m, k);
            double b = deq_row(wq, ws, wc, K, (int64_t)e * N + n, k);
            acc += a * b;
            am += fabs(a * b);
        }
        if (bias) { double bb = orc_bf16_value(bias[(int64_t)e * N + n]); acc += bb; am += fabs(bb); }
        val[i] = acc;
        mag[i] = am;
    }
}

/* dgrad [RQ] [FM]: dX[m,k] = sum_n dY[m,n] * W[e(m),n,k]. dY rowwise (M,N);
 * W colwise: codes (E*N, K) in W's byte order, compact colwise scales of the
 * (E*N, K) matrix (blocks of 32 along n never straddle experts since
 * N % 128 == 0). */
ORC_API void orc_dgrad_entries(const uint8_t* dyq, const uint8_t* dys, const uint8_t* wq, const uint8_t* ws,
                               int64_t M, int64_t N, int64_t K, int E, const int64_t* m_splits,
                               int64_t count, const int64_t* rows, const int64_t* cols, double* val, double* mag) {
    int64_t dr, dc, wr, wc;
    orc_compact_shape(M, N, 0, &dr, &dc);
    orc_compact_shape((int64_t)E * N, K, 1, &wr, &wc);
    #pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = rows[i], k = cols[i];
        int e = expert_of_row(m_splits, E, m, NULL);
        double acc = 0.0, am = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double a = deq_row(dyq, dys, dc, N, m, n);
            double b = deq_col(wq, ws, wc, K, (int64_t)e * N + n, k);
            acc += a * b;
            am += fabs(a * b);
        }
        val[i] = acc;
        mag[i] = am;
    }
}

/* wgrad [RQ] [FM]: dW[e,n,k] = sum over expert e's rows m of dY[m,n]*X[m,k],
 * both from their colwise copies; an empty expert gives 0. Entry i is
 * (experts[i], rows[i] = n, cols[i] = k). */
ORC_API void orc_wgrad_entries(const uint8_t* dyq, const uint8_t* dys, const uint8_t* xq, const uint8_t* xs,
                               int64_t M, int64_t N, int64_t K, int E, const int64_t* m_splits,
                               int64_t count, const int64_t* experts, const int64_t* rows, const int64_t* cols,
                               double* val, double* mag) {
    int64_t dr, dc, xr, xc;
    orc_compact_shape(M, N, 1, &dr, &dc);
    orc_compact_shape(M, K, 1, &xr, &xc);
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i) {
        int e = (int)experts[i];
        int64_t n = rows[i], k = cols[i], off = 0;
        for (int j = 0; j < e; ++j) off += m_splits[j];
        double acc = 0.0, am = 0.0;
        for (int64_t m = off; m < off + m_splits[e]; ++m) {
            double a = deq_col(dyq, dys, dc, N, m, n);
            double b = deq_col(xq, xs, xc, K, m, k);
            acc += a * b;
            am += fabs(a * b);
        }
        val[i] = acc;
        mag[i] = am;
    }
}

/* ----------------------------------------------------------------- SwiGLU */

/* SwiGLU between FC1 and FC2 of the fused grouped MLP [FM]. Reading: the
 * first F columns of the FC1 output are the gate g, the last F the up
 * projection u. h = silu(g) * u, silu(g) = g * sigmoid(g). fp64, rounded
 * once to bf16. */
ORC_API void orc_swiglu_fwd(const uint16_t* y, int64_t M, int64_t F, uint16_t* h) {
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t f = 0; f < F; ++f) {
            double g = orc_bf16_value(y[m * 2 * F + f]);
            double u = orc_bf16_value(y[m * 2 * F + F + f]);
            double sg = 1.0 / (1.0 + exp(-g));
            h[m * F + f] = orc_bf16_round(g * sg * u);
        }
}

/* Backward of SwiGLU: dg = dh * u * sigmoid(g) * (1 + g * (1 - sigmoid(g))),
 * du = dh * silu(g). Output dy (M, 2F) = [dg | du], bf16. */
ORC_API void orc_swiglu_bwd(const uint16_t* dh, const uint16_t* y, int64_t M, int64_t F, uint16_t* dy) {
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t f = 0; f < F; ++f) {
            double d = orc_bf16_value(dh[m * F + f]);
            double g = orc_bf16_value(y[m * 2 * F + f]);
            double u = orc_bf16_value(y[m * 2 * F + F + f]);
            double sg = 1.0 / (1.0 + exp(-g));
            dy[m * 2 * F + f] = orc_bf16_round(d * u * sg * (1.0 + g * (1.0 - sg)));
            dy[m * 2 * F + F + f] = orc_bf16_round(d * g * sg);
        }
}

ORC_API int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
