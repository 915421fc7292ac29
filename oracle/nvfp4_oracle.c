/*
 * CPU oracle for the NVFP4 matmul.  TEST INFRASTRUCTURE ONLY: nothing in the
 * product path may link, load or call this file; only the test suite, the
 * package's smoke check and the benchmark's CPU leg do.
 *
 * The format is named on the "MLX CUDA Cleanup Plan" page (Refactor Plan,
 * Phase 3b: the local checkpoint is mode=nvfp4 with group_size=16, to be run
 * by a CUDA NVFP4 qmv that follows the llama.cpp/ggml modelopt path, kept
 * separate from the affine path).  The page does not spell the format out;
 * the reading used here is the NVFP4 layout as NVIDIA's model optimizer
 * writes it:
 *   - elements are FP4 E2M1 codes (bit 3 sign, bits 2-1 exponent with bias 1,
 *     bit 0 mantissa; exponent 0 is subnormal, value mantissa * 0.5), packed
 *     eight per uint32 word, lowest nibble = lowest k (as the affine codes);
 *   - every 16 consecutive elements along K share one scale stored as FP8
 *     E4M3 (bit 7 sign, bits 6-3 exponent with bias 7, bits 2-0 mantissa;
 *     exponent 0 is subnormal, value mantissa * 2^-9; no infinities,
 *     S.1111.111 is NaN);
 *   - one fp32 scale per tensor multiplies everything (1.0 where a checkpoint
 *     has none).
 * So w[n,k] = global * e4m3(scale[n, k/16]) * e2m1(q[n,k]) and
 * y[m,n] = sum_k x[m,k] * w[n,k], rounded once to bf16 (nearest, ties to
 * even) with aqo_double_to_bf16.
 *
 * Precision: e4m3 * e2m1 has at most 6 significant bits, times the fp32
 * global at most 30: exact in double; x * w (8 more bits) is exact; the
 * k-ordered double sum errs near K * 2^-53.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

uint16_t aqo_double_to_bf16(double v);   /* aq_oracle.c */
double aqo_bf16_to_double(uint16_t h);    /* aq_oracle.c */

double aqo_e2m1_to_double(unsigned code)
{
    const unsigned sign = (code >> 3) & 1u, exp = (code >> 1) & 3u, man = code & 1u;
    double mag;
    if (exp == 0)
        mag = man * 0.5;                              /* subnormal: 0 or 0.5 */
    else
        mag = ldexp(1.0 + man * 0.5, (int)exp - 1);   /* (1 + m/2) * 2^(e - 1) */
    return sign ? -mag : mag;
}

double aqo_e4m3_to_double(unsigned byte)
{
    const unsigned sign = (byte >> 7) & 1u, exp = (byte >> 3) & 15u, man = byte & 7u;
    double mag;
    if (exp == 15 && man == 7)
        return NAN;                                   /* the only non-finite encoding */
    if (exp == 0)
        mag = ldexp((double)man, -9);                 /* subnormal: m/8 * 2^(1 - 7) */
    else
        mag = ldexp(1.0 + man / 8.0, (int)exp - 7);
    return sign ? -mag : mag;
}

static unsigned nibble(const uint32_t *row_words, int64_t k)
{
    return (row_words[k >> 3] >> (4 * (k & 7))) & 15u;
}

/* w[n,k] for the whole matrix, row-major N x K doubles. */
int aqo_nvfp4_dequant(const uint32_t *w_packed, const uint8_t *scales, float global, int64_t N, int64_t K,
                      double *w)
{
    if (N < 0 || K < 0 || K % 16)
        return 1;
    for (int64_t n = 0; n < N; ++n) {
        const uint32_t *rw = w_packed + n * (K / 8);
        const uint8_t *rs = scales + n * (K / 16);
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = (double)global * aqo_e4m3_to_double(rs[k / 16]) * aqo_e2m1_to_double(nibble(rw, k));
    }
    return 0;
}

static double dot(const uint16_t *xm, const uint32_t *rw, const uint8_t *rs, float global, int64_t K)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double w = (double)global * aqo_e4m3_to_double(rs[k / 16]) * aqo_e2m1_to_double(nibble(rw, k));
        acc += aqo_bf16_to_double(xm[k]) * w;
    }
    return acc;
}

int aqo_nvfp4_matmul(const uint16_t *x, const uint32_t *w_packed, const uint8_t *scales, float global, int64_t M,
                     int64_t N, int64_t K, double *y_exact, uint16_t *y_bf16)
{
    if (M < 0 || N < 0 || K < 0 || K % 16)
        return 1;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            const double v = dot(x + m * K, w_packed + n * (K / 8), scales + n * (K / 16), global, K);
            y_exact[m * N + n] = v;
            y_bf16[m * N + n] = aqo_double_to_bf16(v);
        }
    return 0;
}

int aqo_nvfp4_matmul_sampled(const uint16_t *x, const uint32_t *w_packed, const uint8_t *scales, float global,
                             int64_t M, int64_t N, int64_t K, const int64_t *idx_m, const int64_t *idx_n,
                             int64_t count, double *y_exact, uint16_t *y_bf16)
{
    if (M < 0 || N < 0 || K < 0 || K % 16)
        return 1;
    for (int64_t i = 0; i < count; ++i) {
        const int64_t m = idx_m[i], n = idx_n[i];
        if (m < 0 || m >= M || n < 0 || n >= N)
            return 2;
        const double v = dot(x + m * K, w_packed + n * (K / 8), scales + n * (K / 16), global, K);
        y_exact[i] = v;
        y_bf16[i] = aqo_double_to_bf16(v);
    }
    return 0;
}
