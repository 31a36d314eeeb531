/*
 * oracle.c -- plain CPU reference for fine-grained FP8 quantization and the
 * block-scaled FP8 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the parity oracle: it is called by
 * the test-suite, by the smoke check and by the CPU-baseline leg of the
 * benchmark, never by the product path.  It shares no code, header, table or
 * constant generator with the CUDA library, and includes none of its files.
 *
 * Sources (web pages on the DeepSeek-V3 FP8 training scheme, cited by host):
 *   [dssusan]  "dssusan.co.kr Q&A post 93378":
 *              - Figure 7(a) passage: activations are grouped and scaled per
 *                1x128 tile (per token per 128 channels), weights per 128x128
 *                block (per 128 input channels per 128 output channels).
 *              - inner-dimension passage: per-group scaling factors along the
 *                inner dimension K of the GEMM; FP8 accumulation on H800
 *                keeps about 14 bits.
 *              - Figure 7(b) passage: GEMMs take FP8 inputs and produce BF16
 *                or FP32 outputs; partial sums are promoted to FP32.
 *              - E4M3 passage: E4M3 on all tensors; the per-group scales are
 *                multiplied in as the dequantization step.
 *   [kailasan] "kailasan.com recruit post 147436", hardware-suggestion
 *              passage: at the promotion interval the partial results are
 *              multiplied by the scaling factors and added into FP32.
 *   OCP 8-bit floating point specification (E4M3): bias 7, 3 mantissa bits,
 *   largest finite 448, subnormals m * 2^-9, S.1111.111 = NaN, no infinity.
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - scale s = amax / 448, computed as an IEEE binary32 division;
 *   - quantized value q = E4M3(fl32(x / s)): a binary32 division, then
 *     round-to-nearest-even into E4M3 with saturation to +-448;
 *   - a group whose s is 0 (all-zero group) gives s = 0 and signed zeros;
 *   - partial groups at a ragged tensor edge take amax over the elements
 *     that exist;
 *   - dequantized value = decode(q) * s, exact in binary64;
 *   - GEMM reference = sum over k of dequantized products, in binary64.
 *
 * Scale layouts (all "K-group major": the scales of one K group are
 * contiguous over the M or N index):
 *   activation 1x128 : s [K/128][lds],  lds >= M,  s[kb*lds + m]
 *   activation 128x1 : sT[ceil(M/128)][ldsT], ldsT >= K, sT[tb*ldsT + k]
 *   weight 128x128   : s [K/128][lds],  lds >= ceil(N/128), s[kb*lds + nb]
 *
 * Parity of every function here is pinned by tests that do not use this file
 * for their expected values (brute-force nearest-code search, exact integer
 * dot products, closed-form tile invariants).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <float.h>

/* Every float expression below must be evaluated in binary32 (SSE), not in
 * a wider format, or the scale and x/s would be rounded differently. */
_Static_assert(FLT_EVAL_METHOD == 0, "binary32 expressions must be evaluated in binary32");

#define ORACLE_E4M3_MAX 448.0f

/* ---------------------------------------------------------------- BF16 -- */

/* A BF16 value is the top 16 bits of a binary32 value: widening is exact. */
static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* --------------------------------------------------------------- E4M3 -- */

/* Round-half-to-even of a non-negative double, written out. */
static double round_half_even(double x)
{
    double fl = floor(x);
    double frac = x - fl;
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/*
 * E4M3 encoding with round-to-nearest-even and saturation (OCP E4M3 format;
 * E4M3 for all tensors per [dssusan] E4M3 passage).
 *
 * For |v| below the largest finite value, the representable neighbours of
 * |v| are multiples of quantum = 2^(E-3), E = max(floor(log2|v|), -6): that
 * spacing holds for the normal binade [2^E, 2^(E+1)) and for the subnormal
 * range below 2^-6.  |v| / quantum is exact in binary64, so rounding it to an
 * integer n with ties to even gives the nearest code, and n * quantum is the
 * encoded magnitude.  |v| >= 448 saturates to 448 (0x7E): every value there
 * is nearer to 448 than to any other finite code, or past the range.
 */
uint8_t oracle_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (isnan(v)) return (uint8_t)(sign | 0x7F);
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a == 0.0) return sign;

    int e2;
    frexp(a, &e2);              /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;             /* floor(log2 a) */
    if (E < -6) E = -6;         /* subnormal range shares the 2^-9 spacing */
    double quantum = ldexp(1.0, E - 3);
    int n = (int)round_half_even(a / quantum);   /* 0 .. 16 */

    if (E == -6 && n < 8) {
        /* subnormal: exponent field 0, mantissa n, value n * 2^-9 */
        return (uint8_t)(sign | n);
    }
    if (n == 16) {              /* rounding carried into the next binade */
        E += 1;
        n = 8;
    }
    /* normal: value (n/8) * 2^E = (1 + (n-8)/8) * 2^(field-7) */
    int field = E + 7;
    return (uint8_t)(sign | (field << 3) | (n - 8));
}

/* Element-wise encode of an array (for exhaustive tests of the encoder). */
void oracle_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e4m3_encode(v[i]);
}

/* Value of an E4M3 code (OCP E4M3 format), exact in binary64. */
double oracle_e4m3_decode(uint8_t c)
{
    int neg = (c & 0x80) != 0;
    int field = (c >> 3) & 0xF;
    int mant = c & 0x7;
    double mag;
    if (field == 0xF && mant == 0x7) return NAN;
    if (field == 0) mag = ldexp((double)mant, -9);
    else mag = ldexp(1.0 + mant / 8.0, field - 7);
    return neg ? -mag : mag;
}

/* ----------------------------------------------------------- one group -- */

/*
 * Quantize one group of n values (n <= 128, the group being a 1x128 tile, a
 * 128x1 tile or a 128x128 block).  vals[i] are binary32 copies of the BF16
 * inputs.  Online max-abs scaling per group ([dssusan] Figure 7(a) passage:
 * the scale follows the group's own values): s = amax / 448 in binary32.
 */
static float quant_group(const float *vals, int64_t n, uint8_t *codes)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; i++) {
        float a = fabsf(vals[i]);
        if (a > amax) amax = a;
    }
    float s = amax / ORACLE_E4M3_MAX;
    for (int64_t i = 0; i < n; i++) {
        if (s == 0.0f) {
            codes[i] = signbit(vals[i]) ? 0x80 : 0x00;
        } else {
            float y = vals[i] / s;          /* binary32 division */
            codes[i] = oracle_e4m3_encode(y);
        }
    }
    return s;
}

/* --------------------------------------------------------- activations -- */

/*
 * 1x128 activation quantization ([dssusan] Figure 7(a) passage: per token
 * per 128 channels).  x: BF16 bits [M][ldx]; q: [M][K] codes; s[kb*lds + m].
 * K must be a multiple of 128.
 */
void oracle_quant_act_1x128(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                            uint8_t *q, float *s, int64_t lds)
{
    float vals[128];
    uint8_t codes[128];
    for (int64_t m = 0; m < M; m++) {
        for (int64_t kb = 0; kb < K / 128; kb++) {
            for (int64_t i = 0; i < 128; i++)
                vals[i] = bf16_bits_to_float(x[m * ldx + kb * 128 + i]);
            s[kb * lds + m] = quant_group(vals, 128, codes);
            memcpy(q + m * K + kb * 128, codes, 128);
        }
    }
}

/*
 * 128x1 activation quantization: the same rule with the group running along
 * the token index, as needed when activations are kept in FP8 for the
 * weight-gradient GEMM ([dssusan] E4M3 passage: "FP8 Wgrad" keeps the
 * activations in FP8 for the backward pass).  The output is transposed so
 * that tokens become the contiguous (inner, K) index of the Wgrad GEMM:
 * qT: [K][M] codes; sT[tb*ldsT + k] for token group tb = m / 128.  The last
 * token group may be partial (M % 128 != 0): amax over the tokens present.
 */
void oracle_quant_act_128x1(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                            uint8_t *qT, float *sT, int64_t ldsT)
{
    float vals[128];
    uint8_t codes[128];
    for (int64_t k = 0; k < K; k++) {
        for (int64_t tb = 0; tb * 128 < M; tb++) {
            int64_t m0 = tb * 128;
            int64_t n = (M - m0 < 128) ? (M - m0) : 128;
            for (int64_t i = 0; i < n; i++)
                vals[i] = bf16_bits_to_float(x[(m0 + i) * ldx + k]);
            sT[tb * ldsT + k] = quant_group(vals, n, codes);
            for (int64_t i = 0; i < n; i++)
                qT[k * M + m0 + i] = codes[i];
        }
    }
}

/* ------------------------------------------------------------- weights -- */

/*
 * 128x128 weight quantization ([dssusan] Figure 7(a) passage: per 128 input
 * channels per 128 output channels).  w: BF16 bits [N][ldw]; q: [N][K];
 * s[kb*lds + nb].  N may be ragged: the last block row holds N % 128 rows.
 */
void oracle_quant_w_128x128(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                            uint8_t *q, float *s, int64_t lds)
{
    float *vals = (float *)malloc(128 * 128 * sizeof(float));
    uint8_t *codes = (uint8_t *)malloc(128 * 128);
    for (int64_t nb = 0; nb * 128 < N; nb++) {
        int64_t n0 = nb * 128;
        int64_t rows = (N - n0 < 128) ? (N - n0) : 128;
        for (int64_t kb = 0; kb < K / 128; kb++) {
            for (int64_t r = 0; r < rows; r++)
                for (int64_t i = 0; i < 128; i++)
                    vals[r * 128 + i] = bf16_bits_to_float(w[(n0 + r) * ldw + kb * 128 + i]);
            s[kb * lds + nb] = quant_group(vals, rows * 128, codes);
            for (int64_t r = 0; r < rows; r++)
                memcpy(q + (n0 + r) * K + kb * 128, codes + r * 128, 128);
        }
    }
    free(vals);
    free(codes);
}

/* ---------------------------------------------------------------- GEMM -- */

/*
 * Block-scaled FP8 GEMM reference, C = A * B^T on dequantized values
 * ([dssusan] inner-dimension and E4M3 passages: per-group scales along K,
 * applied as the dequantization; [kailasan] hardware-suggestion passage:
 * each partial result is multiplied by its scaling factors and summed in
 * FP32 -- here the sum is taken in binary64, the exact-up-to-rounding value
 * that any promotion interval approximates).
 *
 *   a_hat[m][k] = decode(A[m*K + k]) * sa[kb*lda_s + m]
 *   b_hat[n][k] = decode(B[n*K + k]) * sb[kb*ldb_s + n/128]   (bkind 0, 128x128)
 *               = decode(B[n*K + k]) * sb[kb*ldb_s + n]       (bkind 1, per row)
 *   C[r][n] = sum_k a_hat[m][k] * b_hat[n][k],  S[r][n] = sum_k |a_hat * b_hat|
 *
 * for each requested row m = rows[r] (rows == NULL: all M rows in order).
 * S is the magnitude sum the error bound is stated in.
 */
void oracle_gemm_blockscaled(const uint8_t *A, const float *sa, int64_t lda_s,
                             const uint8_t *B, const float *sb, int64_t ldb_s, int bkind,
                             int64_t M, int64_t N, int64_t K,
                             const int64_t *rows, int64_t nrows,
                             double *C, double *S)
{
    int64_t nr = rows ? nrows : M;
    double *ahat = (double *)malloc((size_t)K * sizeof(double));
    for (int64_t r = 0; r < nr; r++) {
        int64_t m = rows ? rows[r] : r;
        for (int64_t k = 0; k < K; k++)
            ahat[k] = oracle_e4m3_decode(A[m * K + k]) * (double)sa[(k / 128) * lda_s + m];
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; k++) {
                int64_t sidx = (k / 128) * ldb_s + (bkind == 0 ? n / 128 : n);
                double bhat = oracle_e4m3_decode(B[n * K + k]) * (double)sb[sidx];
                double p = ahat[k] * bhat;
                acc += p;
                mag += fabs(p);
            }
            C[r * N + n] = acc;
            S[r * N + n] = mag;
        }
    }
    free(ahat);
}

/*
 * Grouped (MoE, contiguous layout) reference: row m of A belongs to expert
 * e = m_indices[m]; e < 0 marks a padding row, whose output is not defined
 * (written as NaN with S = 0 here).  B: [E][N][K] codes;
 * sb: [E][K/128][ldb_s] 128x128 block scales, one stack per expert.
 */
void oracle_grouped_gemm_blockscaled(const uint8_t *A, const float *sa, int64_t lda_s,
                                     const uint8_t *B, const float *sb, int64_t ldb_s,
                                     const int32_t *m_indices, int32_t num_experts,
                                     int64_t M, int64_t N, int64_t K,
                                     const int64_t *rows, int64_t nrows,
                                     double *C, double *S)
{
    int64_t nr = rows ? nrows : M;
    int64_t KB = K / 128;
    for (int64_t r = 0; r < nr; r++) {
        int64_t m = rows ? rows[r] : r;
        int32_t e = m_indices[m];
        if (e < 0 || e >= num_experts) {
            for (int64_t n = 0; n < N; n++) {
                C[r * N + n] = NAN;
                S[r * N + n] = 0.0;
            }
            continue;
        }
        int64_t one = m;
        /* one row of the dense reference against expert e's weights */
        oracle_gemm_blockscaled(A, sa, lda_s,
                                B + (int64_t)e * N * K, sb + (int64_t)e * KB * ldb_s, ldb_s, 0,
                                M, N, K, &one, 1, C + r * N, S + r * N);
    }
}

/* -------------------------------------------------- accumulation probe -- */

/*
 * Exact dot product of two E4M3 code vectors.  Every finite E4M3 value is an
 * integer multiple of 2^-9 with |value| <= 448 = 229376 * 2^-9, so every
 * product is an integer multiple of 2^-18 below 2^36 * 2^-18, and a sum of up
 * to 2^26 products fits in a signed 64-bit integer.  Returns the sum in units
 * of 2^-18 (the caller scales by 2^-18).  Used to measure how many bits the
 * tensor-core accumulation keeps ([dssusan] inner-dimension passage: about
 * 14 bits on H800).
 */
int64_t oracle_dot_e4m3_exact(const uint8_t *a, const uint8_t *b, int64_t K)
{
    int64_t acc = 0;
    for (int64_t k = 0; k < K; k++) {
        double va = oracle_e4m3_decode(a[k]) * 512.0;   /* exact integer */
        double vb = oracle_e4m3_decode(b[k]) * 512.0;
        acc += (int64_t)va * (int64_t)vb;
    }
    return acc;
}
