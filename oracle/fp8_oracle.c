/*
 * fp8_oracle.c -- plain, slow, CPU-only oracle for the fine-grained FP8 GEMM path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * loads this file; only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg may.  It shares no code, header or table with the CUDA path.
 *
 * What it computes, and where the pages say so:
 *   - Activations are quantised per 1x128 tile (one scale per row per 128
 *     K-columns), weights per 128x128 block.
 *     ["DeepSeek-V3 training walkthrough" (deepseek.csdn.net), section
 *      二(四) "FP8 low-precision training", fine-grained quantisation item;
 *      "DeepSeek-V3 Technical Report digest" (sherconan.github.io), section 3
 *      "FP8 mixed-precision training", fine-grained quantisation bullet;
 *      qqstock.cn walkthrough, FP8 section, report figure 7a.]
 *   - Every 128 accumulated K-elements the partial product is promoted to FP32
 *     and the two scales are applied; all three GEMM kinds use FP8.
 *     [Technical Report digest, section 3, "precision promotion" and
 *      "FP8 operations" bullets; walkthrough 二(四), MMA-into-FP32 item;
 *      qqstock.cn walkthrough, report figure 7b.]
 *   The pages fix neither the FP8 format, nor the scale formula, nor rounding.
 *   The readings taken here (E4M3 "FN", scale = amax/448 as one IEEE fp32
 *   division, q = E4M3_RNE_satfinite(fp32(x / scale)), zero block -> scale 0)
 *   are the plainest ones and are listed with the others in the design notes.
 *
 * Every function is the definition written out: no blocking, no reordering.
 * The GEMMs spread whole output rows over OpenMP threads; every output
 * element is one in-order sum over k on one thread, so the thread count does
 * not change any result.
 * Floating-point environment: IEEE-754 binary32/binary64, round-to-nearest,
 * no flush-to-zero (x86-64 SSE arithmetic; compiled without fast-math).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* bf16 -> fp32: a bf16 value is the top 16 bits of the binary32 pattern.    */
static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a non-negative double to the nearest integer, ties to even.
 * Written out instead of relying on the current rounding mode. */
static double round_half_even_nonneg(double x)
{
    double f = floor(x);
    double d = x - f;              /* exact for the magnitudes used here */
    if (d > 0.5) return f + 1.0;
    if (d < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* ------------------------------------------------------------------------ */
/* E4M3 ("FN" variant of the OCP 8-bit floating-point formats): 1 sign bit,
 * 4 exponent bits (bias 7), 3 mantissa bits; no infinities; S.1111.111 is NaN;
 * largest finite magnitude S.1111.110 = 448; smallest normal 2^-6; subnormals
 * m/8 * 2^-6.
 *
 * encode: round-to-nearest-even with saturation to +-448 (the "satfinite"
 * reading).  Input must be finite.  The sign bit of the input is kept, so
 * -0.0 encodes as 0x80 and a negative value that rounds to zero as 0x80.     */
uint8_t oracle_e4m3_encode(float v)
{
    uint32_t bits;
    memcpy(&bits, &v, sizeof bits);
    const uint8_t sign = (bits >> 31) ? 0x80u : 0x00u;
    const double a = fabs((double)v);          /* exact */

    if (a >= 448.0)
        return (uint8_t)(sign | 0x7Eu);        /* saturate to the largest finite */

    if (a < ldexp(1.0, -6)) {
        /* subnormal range: value = m * 2^-9, m in [0, 8]; a * 2^9 is exact.
         * m == 8 is 2^-6, whose code 0x08 is the smallest normal. */
        double m = round_half_even_nonneg(a * 512.0);
        return (uint8_t)(sign | (uint8_t)m);
    }

    int e2;
    (void)frexp(a, &e2);                       /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                            /* floor(log2 a), in [-6, 8]    */
    /* a * 2^(3-e) lies in [8, 16); rounding it to an integer keeps 4
     * significant bits, i.e. 1 implicit + 3 mantissa bits. */
    double m = round_half_even_nonneg(ldexp(a, 3 - e)) - 8.0;
    if (m == 8.0) {                            /* rounded up into the next binade */
        e += 1;
        m = 0.0;
    }
    /* a < 448 keeps (e, m) <= (8, 6): code S.1111.110 at most. */
    return (uint8_t)(sign | (uint8_t)(((e + 7) << 3) | (int)m));
}

int oracle_get_threads(void);

/* encode over an array (for exhaustive checks of the encoder).  Elements are
 * independent; the loop is spread over the oracle's threads (no change to
 * any element's arithmetic). */
void oracle_e4m3_encode_n(const float *v, int64_t n, uint8_t *out)
{
#pragma omp parallel for schedule(static) num_threads(oracle_get_threads())
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(v[i]);
}

/* decode: (-1)^s * 2^(E-7) * (1 + m/8) for E >= 1, (-1)^s * 2^-6 * m/8 for E == 0. */
double oracle_e4m3_decode(uint8_t c)
{
    const int s = c >> 7;
    const int E = (c >> 3) & 0xF;
    const int m = c & 0x7;
    if (E == 15 && m == 7)
        return NAN;
    double v = (E == 0) ? ldexp((double)m / 8.0, -6)
                        : ldexp(1.0 + (double)m / 8.0, E - 7);
    return s ? -v : v;
}

/* One quantisation group (a 1x128 tile or a 128x128 block), given its amax.
 * scale = fp32(amax / 448) -- one IEEE binary32 division.
 * q     = encode(fp32(x / scale)) -- one IEEE binary32 division per element.
 * amax == 0 (the group is all +-0): scale = 0 and each code is encode(x),
 * which keeps the sign of the zero. */
static float group_scale(float amax)
{
    return amax / 448.0f;
}

static uint8_t quantise_element(float x, float scale)
{
    if (scale == 0.0f)
        return oracle_e4m3_encode(x);
    float y = x / scale;
    return oracle_e4m3_encode(y);
}

/* ------------------------------------------------------------------------ */
/* 1x128 activation quantiser.
 *   x  : bf16 bits, row-major [M][K], row stride ldx (elements)
 *   q  : E4M3 codes, row-major [M][K], row stride ldq (bytes)
 *   sA : fp32 scales, [K/128][M] (M contiguous)
 * Returns 0, or -2 when K is not a multiple of 128. */
int oracle_quant_act_1x128(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                           uint8_t *q, int64_t ldq, float *sA)
{
    if (K % 128 != 0)
        return -2;
    const int64_t KB = K / 128;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f;
            for (int64_t k = kb * 128; k < kb * 128 + 128; ++k) {
                float a = fabsf(bf16_bits_to_float(x[m * ldx + k]));
                if (a > amax)
                    amax = a;
            }
            float s = group_scale(amax);
            sA[kb * M + m] = s;
            for (int64_t k = kb * 128; k < kb * 128 + 128; ++k)
                q[m * ldq + k] = quantise_element(bf16_bits_to_float(x[m * ldx + k]), s);
        }
    }
    return 0;
}

/* 128x128 weight quantiser.
 *   w  : bf16 bits, row-major [R][C], row stride ldw (elements)
 *   q  : E4M3 codes, row-major [R][C], row stride ldq (bytes)
 *   sW : fp32 scales, [ceil(R/128)][C/128] row-major
 * A last row-block with fewer than 128 rows takes its amax over the rows that
 * exist.  Returns 0, or -2 when C is not a multiple of 128. */
int oracle_quant_w_128x128(const uint16_t *w, int64_t R, int64_t C, int64_t ldw,
                           uint8_t *q, int64_t ldq, float *sW)
{
    if (C % 128 != 0)
        return -2;
    const int64_t RB = (R + 127) / 128, CB = C / 128;
    for (int64_t rb = 0; rb < RB; ++rb) {
        const int64_t r1 = (rb * 128 + 128 < R) ? rb * 128 + 128 : R;
        for (int64_t cb = 0; cb < CB; ++cb) {
            float amax = 0.0f;
            for (int64_t r = rb * 128; r < r1; ++r)
                for (int64_t c = cb * 128; c < cb * 128 + 128; ++c) {
                    float a = fabsf(bf16_bits_to_float(w[r * ldw + c]));
                    if (a > amax)
                        amax = a;
                }
            float s = group_scale(amax);
            sW[rb * CB + cb] = s;
            for (int64_t r = rb * 128; r < r1; ++r)
                for (int64_t c = cb * 128; c < cb * 128 + 128; ++c)
                    q[r * ldq + c] = quantise_element(bf16_bits_to_float(w[r * ldw + c]), s);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Threads.  The GEMMs below split their OUTPUT ROWS over OpenMP threads; each
 * output element is still one sum over k = 0, 1, ..., K-1 in that order, on
 * one thread, so the result does not depend on the thread count (pinned by a
 * test that compares 1 thread with many).  0 = the OpenMP default. */
static int g_threads = 0;

void oracle_set_threads(int n) { g_threads = n < 0 ? 0 : n; }

int oracle_get_threads(void)
{
#ifdef _OPENMP
    return g_threads > 0 ? g_threads : omp_get_max_threads();
#else
    return 1;
#endif
}

/* Value of every code, from oracle_e4m3_decode: filled once, before any
 * parallel loop reads it. */
static double g_dec[256];
static int g_dec_ready = 0;

static void dec_table_init(void)
{
    if (g_dec_ready)
        return;
    for (int c = 0; c < 256; ++c)
        g_dec[c] = oracle_e4m3_decode((uint8_t)c);
    g_dec_ready = 1;
}

/* ------------------------------------------------------------------------ */
/* Dequantised operands, float64 (each value dec(q) * scale is exact: a 4-bit
 * by 24-bit significand product). */
static double deq_a(const uint8_t *qA, const float *sA, int64_t M, int64_t lda,
                    int64_t m, int64_t k)
{
    return g_dec[qA[m * lda + k]] * (double)sA[(k / 128) * M + m];
}

/* B element (n, k) of the GEMM's B^T operand.
 * b_major 0: qB stored [N][K] (row stride ldb), sB [ceil(N/128)][K/128].
 * b_major 1: qB stored [K][N] (row stride ldb), sB [K/128][ceil(N/128)]. */
static double deq_b(const uint8_t *qB, const float *sB, int64_t N, int64_t K,
                    int64_t ldb, int b_major, int64_t n, int64_t k)
{
    const int64_t KB = K / 128, NB = (N + 127) / 128;
    if (b_major == 0)
        return g_dec[qB[n * ldb + k]] * (double)sB[(n / 128) * KB + k / 128];
    return g_dec[qB[k * ldb + n]] * (double)sB[(k / 128) * NB + n / 128];
}

/* C[m][n] = sum_k A^[m][k] * B^[n][k], in float64, over the dequantised
 * operands.  This is the result the block-scaled GEMM defines: per 128-wide
 * K-slice the FP8 product is scaled by sA * sB and summed in higher precision;
 * summing dequantised products gives the same exact-arithmetic value.
 * Row m's dequantised values A^[m][0..K) are formed once into `arow` and
 * reused for every n (the same numbers deq_a returns). */
int oracle_gemm_f64(const uint8_t *qA, const float *sA, int64_t lda,
                    const uint8_t *qB, const float *sB, int64_t ldb, int b_major,
                    int64_t M, int64_t N, int64_t K, double *C, int64_t ldc)
{
    if (K % 128 != 0)
        return -2;
    dec_table_init();
    int fail = 0;
#pragma omp parallel num_threads(oracle_get_threads())
    {
        double *arow = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        if (!arow) {
#pragma omp atomic write
            fail = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t m = 0; m < M; ++m) {
            if (!arow)
                continue;
            for (int64_t k = 0; k < K; ++k)
                arow[k] = deq_a(qA, sA, M, lda, m, k);
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += arow[k] * deq_b(qB, sB, N, K, ldb, b_major, n, k);
                C[m * ldc + n] = acc;
            }
        }
        free(arow);
    }
    return fail ? -5 : 0;
}

/* The same sum at `count` chosen (row, col) positions, for sampled checks of
 * shapes too large to compute in full. */
int oracle_gemm_f64_at(const uint8_t *qA, const float *sA, int64_t lda,
                       const uint8_t *qB, const float *sB, int64_t ldb, int b_major,
                       int64_t M, int64_t N, int64_t K,
                       const int64_t *rows, const int64_t *cols, int64_t count, double *out)
{
    if (K % 128 != 0)
        return -2;
    for (int64_t i = 0; i < count; ++i)
        if (rows[i] < 0 || rows[i] >= M || cols[i] < 0 || cols[i] >= N)
            return -4;
    dec_table_init();
#pragma omp parallel for schedule(dynamic, 16) num_threads(oracle_get_threads())
    for (int64_t i = 0; i < count; ++i) {
        const int64_t m = rows[i], n = cols[i];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += deq_a(qA, sA, M, lda, m, k) * deq_b(qB, sB, N, K, ldb, b_major, n, k);
        out[i] = acc;
    }
    return 0;
}

/* Grouped GEMM for routed experts: rows [off[e], off[e+1]) of A belong to
 * expert e, whose weight is qB[e] ([N][K] per expert, K contiguous) with
 * scales sB[e] ([ceil(N/128)][K/128]).  C is [M_total][N].
 * Experts: 256 routed, top-8 per token ["DeepSeek-V3 training walkthrough",
 * section 一 architecture, DeepSeekMoE item]. */
int oracle_grouped_gemm_f64(const uint8_t *qA, const float *sA, int64_t lda,
                            const uint8_t *qB, const float *sB,
                            const int32_t *off, int E, int64_t M_total,
                            int64_t N, int64_t K, double *C, int64_t ldc)
{
    if (K % 128 != 0)
        return -2;
    dec_table_init();
    const int64_t NB = (N + 127) / 128, KB = K / 128;
    for (int e = 0; e < E; ++e) {
        const uint8_t *qBe = qB + (int64_t)e * N * K;
        const float *sBe = sB + (int64_t)e * NB * KB;
#pragma omp parallel for schedule(dynamic, 1) num_threads(oracle_get_threads())
        for (int64_t m = off[e]; m < off[e + 1]; ++m)
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += deq_a(qA, sA, M_total, lda, m, k) * deq_b(qBe, sBe, N, K, K, 0, n, k);
                C[m * ldc + n] = acc;
            }
    }
    return 0;
}

/* Weight-gradient GEMM, both operands quantised per 1x128 tile along the
 * contraction dimension (the token dimension of dW = dY^T . X): A is [M][K]
 * with sA [K/128][M] and B is [N][K] with sB [K/128][N] -- each B row carries
 * its own scale per 128-wide K-slice, exactly like an activation row.
 *   C[m][n] = sum_k A^[m][k] * B^[n][k]  (float64 over dequantised operands)
 * ["DeepSeek-V3 Technical Report digest", section 3, "FP8 operations" bullet:
 *  forward, data-gradient and weight-gradient GEMMs all run in FP8;
 *  fine-grained 1x128 tiles for activation-like operands.] */
int oracle_gemm_f64_tokens(const uint8_t *qA, const float *sA, int64_t lda,
                           const uint8_t *qB, const float *sB, int64_t ldb,
                           int64_t M, int64_t N, int64_t K, double *C, int64_t ldc)
{
    if (K % 128 != 0)
        return -2;
    dec_table_init();
#pragma omp parallel for schedule(dynamic, 1) num_threads(oracle_get_threads())
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += deq_a(qA, sA, M, lda, m, k) * deq_a(qB, sB, N, ldb, n, k);
            C[m * ldc + n] = acc;
        }
    return 0;
}

/* Euclidean norms of the dequantised rows, used to normalise the GEMM error:
 * act: ||A^[m,:]||_2 for each m;  b: ||B^[n,:]||_2 for each n (B^ as above). */
void oracle_act_row_norms(const uint8_t *qA, const float *sA, int64_t lda,
                          int64_t M, int64_t K, double *out)
{
    dec_table_init();
#pragma omp parallel for schedule(static) num_threads(oracle_get_threads())
    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double v = deq_a(qA, sA, M, lda, m, k);
            ss += v * v;
        }
        out[m] = sqrt(ss);
    }
}

void oracle_b_row_norms(const uint8_t *qB, const float *sB, int64_t ldb, int b_major,
                        int64_t N, int64_t K, double *out)
{
    dec_table_init();
#pragma omp parallel for schedule(static) num_threads(oracle_get_threads())
    for (int64_t n = 0; n < N; ++n) {
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double v = deq_b(qB, sB, N, K, ldb, b_major, n, k);
            ss += v * v;
        }
        out[n] = sqrt(ss);
    }
}

/* ------------------------------------------------------------------------ */
/* Per-tensor scaling: the contrast to the fine-grained scheme.  The pages
 * describe their 1x128 / 128x128 groups as finer than scaling a whole tensor
 * by one factor, which lets a few outliers set the scale of every element
 * [qqstock.cn walkthrough, FP8 section: fine-grained rather than per-tensor
 * quantisation; "DeepSeek-V3 Technical Report digest", section 3,
 * fine-grained quantisation bullet].  The same rules apply with the group
 * being the whole tensor: scale = fp32(amax / 448), q = enc(fp32(x / scale)),
 * an all-zero tensor gets scale 0 and codes enc(x).                          */
static float tensor_amax(const uint16_t *x, int64_t R, int64_t C, int64_t ldx)
{
    float amax = 0.0f;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            float a = fabsf(bf16_bits_to_float(x[r * ldx + c]));
            if (a > amax)
                amax = a;
        }
    return amax;
}

/* Current scaling: the scale comes from this tensor's own amax. */
int oracle_quant_per_tensor(const uint16_t *x, int64_t R, int64_t C, int64_t ldx,
                            uint8_t *q, int64_t ldq, float *scale)
{
    const float s = group_scale(tensor_amax(x, R, C, ldx));
    *scale = s;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c)
            q[r * ldq + c] = quantise_element(bf16_bits_to_float(x[r * ldx + c]), s);
    return 0;
}

/* Delayed scaling: the scale comes from an amax given by the caller (the
 * largest amax of earlier steps), s = fp32(amax_in / 448); values beyond
 * 448 * s saturate to +-448.  Also returns this tensor's amax, the value a
 * caller records for later steps. */
int oracle_quant_per_tensor_delayed(const uint16_t *x, int64_t R, int64_t C, int64_t ldx,
                                    float amax_in, uint8_t *q, int64_t ldq, float *scale,
                                    float *amax_out)
{
    const float s = group_scale(amax_in);
    *scale = s;
    *amax_out = tensor_amax(x, R, C, ldx);
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c)
            q[r * ldq + c] = quantise_element(bf16_bits_to_float(x[r * ldx + c]), s);
    return 0;
}

/* GEMM over per-tensor quantised operands:
 *   C[m][n] = sum_k dec(qA[m][k]) * sA * dec(qB(n, k)) * sB   (float64)
 * qB is [N][K] (b_major 0) or stored [K][N] (b_major 1). */
int oracle_gemm_f64_per_tensor(const uint8_t *qA, float sA, int64_t lda,
                               const uint8_t *qB, float sB, int64_t ldb, int b_major,
                               int64_t M, int64_t N, int64_t K, double *C, int64_t ldc)
{
    dec_table_init();
#pragma omp parallel for schedule(dynamic, 1) num_threads(oracle_get_threads())
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const uint8_t b = b_major == 0 ? qB[n * ldb + k] : qB[k * ldb + n];
                acc += g_dec[qA[m * lda + k]] * (double)sA * (g_dec[b] * (double)sB);
            }
            C[m * ldc + n] = acc;
        }
    return 0;
}

/* The unquantised product of the BF16 inputs, in float64:
 *   C[m][n] = sum_k a[m][k] * b(n, k)
 * (b [N][K] for b_major 0, stored [K][N] for b_major 1).  It is the value
 * both FP8 schemes approximate; the pages judge FP8 training against BF16
 * ["DeepSeek-V3 Technical Report digest", section 3: relative loss error of
 * FP8 against BF16 below 0.25%]. */
int oracle_gemm_bf16_f64(const uint16_t *a, int64_t lda, const uint16_t *b, int64_t ldb, int b_major,
                         int64_t M, int64_t N, int64_t K, double *C, int64_t ldc)
{
#pragma omp parallel for schedule(dynamic, 1) num_threads(oracle_get_threads())
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const uint16_t bb = b_major == 0 ? b[n * ldb + k] : b[k * ldb + n];
                acc += (double)bf16_bits_to_float(a[m * lda + k]) * (double)bf16_bits_to_float(bb);
            }
            C[m * ldc + n] = acc;
        }
    return 0;
}
