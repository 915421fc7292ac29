/*
 * CPU oracle for the affine group-quantized matmul.  TEST INFRASTRUCTURE ONLY:
 * nothing in the product path may link, load or call this file; only the test
 * suite, the package's smoke check and the benchmark's CPU-baseline leg do.
 *
 * What it computes is the plain definition, written out with no blocking,
 * fusion or reordering:
 *
 *   y[m,n] = sum_k x[m,k] * w[n,k],   w[n,k] = scale[n,k/gs] * q[n,k] + bias[n,k/gs]
 *
 * Operand types follow "MLX CUDA Cleanup Plan", Target Architecture section 1:
 * bf16 activations, weights packed into 32-bit words, bf16 scales and biases;
 * 4-bit and 8-bit affine packed weights with group size 64 are the variants its
 * Refactor Plan, Phase 3, lists.  The pages do not print the
 * bit layout or the dequantization formula; the readings used here are:
 *   - codes are unsigned, (32/bits) per uint32 word, the lowest bits holding
 *     the lowest k ("low nibble first along K" for 4-bit);
 *   - groups run along K, contiguous, never straddling a row;
 *   - dequantization is scale*q + bias.
 * Results are rounded once, from double, to bf16 (nearest, ties to even):
 * the Verification Requirements section of the same page asks that results
 * follow bf16 rounding.
 *
 * Precision: every bf16 value widens to double exactly; scale*q + bias is
 * exact in double for the value ranges used (a 12-bit product plus an 8-bit
 * significand); x*w is exact (8 x <= 25 bits); the k-ordered double sum has a
 * relative error near K*2^-53, far below one bf16 ulp.
 *
 * Every function is pinned by the CPU tests (pack/unpack round trip, nibble
 * order fixture, dequantization endpoints, one-hot and zero inputs, a closed
 * form, exact rational brute force on tiny shapes, exhaustive bf16 rounding).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---- bf16 <-> double -------------------------------------------------- */

double aqo_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), directly from double so
 * that no intermediate float rounding happens.  bf16 has 8 significant bits
 * and the float32 exponent range: the spacing of representable values around
 * |v| is 2^(e-7) for 2^e <= |v| < 2^(e+1), and 2^-133 below 2^-126
 * (subnormals).  Scaling by a power of two is exact, so v/spacing is rounded
 * to an integer with rint() (the default rounding mode is nearest-even). */
uint16_t aqo_double_to_bf16(double v)
{
    if (isnan(v))
        return (uint16_t)(signbit(v) ? 0xFFC0u : 0x7FC0u);
    if (isinf(v))
        return (uint16_t)(signbit(v) ? 0xFF80u : 0x7F80u);
    if (v == 0.0)
        return (uint16_t)(signbit(v) ? 0x8000u : 0x0000u);
    int e2;
    frexp(v, &e2);          /* |v| = f * 2^e2, f in [0.5, 1): 2^(e2-1) <= |v| < 2^e2 */
    int e = e2 - 1;         /* 2^e <= |v| < 2^(e+1) */
    if (e < -126)
        e = -126;           /* subnormal range shares the spacing of the smallest binade */
    double spacing = ldexp(1.0, e - 7);
    double r = rint(v / spacing) * spacing;
    if (fabs(r) >= ldexp(1.0, 128))
        return (uint16_t)(signbit(v) ? 0xFF80u : 0x7F80u);
    float f = (float)r;     /* exact: r is representable in bf16, hence in float */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

void aqo_double_to_bf16_array(const double *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = aqo_double_to_bf16(v[i]);
}

/* ---- packing ---------------------------------------------------------- */

/* Code k of row n: bits [bits*(k mod per), bits*(k mod per) + bits) of word
 * k / per of that row, per = 32/bits codes per word. */
static unsigned code_at(const uint32_t *row_words, int64_t k, int bits)
{
    int per = 32 / bits;
    uint32_t word = row_words[k / per];
    int shift = bits * (int)(k % per);
    uint32_t mask = (bits == 32) ? 0xFFFFFFFFu : ((1u << bits) - 1u);
    return (unsigned)((word >> shift) & mask);
}

int aqo_unpack(const uint32_t *w_packed, int64_t N, int64_t K, int bits, uint8_t *codes)
{
    if (bits != 4 && bits != 8)
        return 1;
    int64_t words = K * bits / 32;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            codes[n * K + k] = (uint8_t)code_at(w_packed + n * words, k, bits);
    return 0;
}

int aqo_pack(const uint8_t *codes, int64_t N, int64_t K, int bits, uint32_t *w_packed)
{
    if (bits != 4 && bits != 8)
        return 1;
    int per = 32 / bits;
    int64_t words = K * bits / 32;
    memset(w_packed, 0, (size_t)(N * words) * sizeof(uint32_t));
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            uint32_t c = codes[n * K + k] & ((1u << bits) - 1u);
            w_packed[n * words + k / per] |= c << (bits * (int)(k % per));
        }
    return 0;
}

/* ---- dequantization --------------------------------------------------- */

/* w[n,k] = scale[n,g] * q[n,k] + bias[n,g], g = k / group_size, in double. */
static void dequant_row(const uint32_t *row_words, const uint16_t *row_s, const uint16_t *row_b,
                        int64_t K, int group_size, int bits, double *w)
{
    for (int64_t k = 0; k < K; ++k) {
        int64_t g = k / group_size;
        double s = aqo_bf16_to_double(row_s[g]);
        double b = aqo_bf16_to_double(row_b[g]);
        w[k] = s * (double)code_at(row_words, k, bits) + b;
    }
}

int aqo_dequant(const uint32_t *w_packed, const uint16_t *scales, const uint16_t *biases,
                int64_t N, int64_t K, int group_size, int bits, double *w)
{
    if ((bits != 4 && bits != 8) || group_size <= 0 || K % group_size)
        return 1;
    int64_t words = K * bits / 32, G = K / group_size;
    for (int64_t n = 0; n < N; ++n)
        dequant_row(w_packed + n * words, scales + n * G, biases + n * G, K, group_size, bits,
                    w + n * K);
    return 0;
}

/* ---- matmul ----------------------------------------------------------- */

typedef struct {
    const uint16_t *x;
    const uint32_t *w_packed;
    const uint16_t *scales, *biases;
    int64_t M, N, K;
    int group_size, bits;
    /* full mode: all (m, n); sampled mode: count pairs from idx_m / idx_n */
    const int64_t *idx_m, *idx_n;
    int64_t count;
    double *y_exact;
    uint16_t *y_bf16;
    int nthreads, tid;
} job_t;

static double dot_row(const uint16_t *xm, const double *w, int64_t K)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k)
        acc += aqo_bf16_to_double(xm[k]) * w[k];
    return acc;
}

static void *full_worker(void *arg)
{
    job_t *j = (job_t *)arg;
    int64_t words = j->K * j->bits / 32, G = j->K / j->group_size;
    double *w = (double *)malloc((size_t)j->K * sizeof(double));
    if (!w)
        return (void *)1;
    /* rows n are dealt out round-robin; each row is dequantized once and
     * dotted with every x row */
    for (int64_t n = j->tid; n < j->N; n += j->nthreads) {
        dequant_row(j->w_packed + n * words, j->scales + n * G, j->biases + n * G, j->K,
                    j->group_size, j->bits, w);
        for (int64_t m = 0; m < j->M; ++m) {
            double v = dot_row(j->x + m * j->K, w, j->K);
            if (j->y_exact)
                j->y_exact[m * j->N + n] = v;
            if (j->y_bf16)
                j->y_bf16[m * j->N + n] = aqo_double_to_bf16(v);
        }
    }
    free(w);
    return NULL;
}

static void *sampled_worker(void *arg)
{
    job_t *j = (job_t *)arg;
    int64_t words = j->K * j->bits / 32, G = j->K / j->group_size;
    double *w = (double *)malloc((size_t)j->K * sizeof(double));
    if (!w)
        return (void *)1;
    for (int64_t i = j->tid; i < j->count; i += j->nthreads) {
        int64_t m = j->idx_m[i], n = j->idx_n[i];
        dequant_row(j->w_packed + n * words, j->scales + n * G, j->biases + n * G, j->K,
                    j->group_size, j->bits, w);
        double v = dot_row(j->x + m * j->K, w, j->K);
        if (j->y_exact)
            j->y_exact[i] = v;
        if (j->y_bf16)
            j->y_bf16[i] = aqo_double_to_bf16(v);
    }
    free(w);
    return NULL;
}

int aqo_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int run_jobs(job_t *proto, int nthreads, void *(*fn)(void *))
{
    if (nthreads <= 0)
        nthreads = aqo_default_threads();
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return 2;
    }
    int rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].nthreads = nthreads;
        jobs[t].tid = t;
        if (pthread_create(&th[t], NULL, fn, &jobs[t]) != 0) {
            /* run the remaining shares inline */
            for (int u = t; u < nthreads; ++u) {
                jobs[u] = *proto;
                jobs[u].nthreads = nthreads;
                jobs[u].tid = u;
                if (fn(&jobs[u]))
                    rc = 2;
            }
            nthreads = t;
            break;
        }
    }
    for (int t = 0; t < nthreads; ++t) {
        void *ret = NULL;
        pthread_join(th[t], &ret);
        if (ret)
            rc = 2;
    }
    free(jobs);
    free(th);
    return rc;
}

static int check_args(int64_t M, int64_t N, int64_t K, int group_size, int bits)
{
    if (M < 0 || N < 0 || K < 0 || group_size <= 0 || (bits != 4 && bits != 8))
        return 1;
    if (K % group_size || (K * bits) % 32)
        return 1;
    return 0;
}

/* y_exact (double, may be NULL) and y_bf16 (may be NULL) are [M, N] row-major. */
int aqo_matmul(const uint16_t *x, const uint32_t *w_packed, const uint16_t *scales,
               const uint16_t *biases, int64_t M, int64_t N, int64_t K, int group_size, int bits,
               double *y_exact, uint16_t *y_bf16, int nthreads)
{
    if (check_args(M, N, K, group_size, bits))
        return 1;
    job_t j = {x, w_packed, scales, biases, M, N, K, group_size, bits, NULL, NULL, 0,
               y_exact, y_bf16, 0, 0};
    return run_jobs(&j, nthreads, full_worker);
}

/* The same definition evaluated at count (m, n) pairs; outputs are [count]. */
int aqo_matmul_sampled(const uint16_t *x, const uint32_t *w_packed, const uint16_t *scales,
                       const uint16_t *biases, int64_t M, int64_t N, int64_t K, int group_size,
                       int bits, const int64_t *idx_m, const int64_t *idx_n, int64_t count,
                       double *y_exact, uint16_t *y_bf16, int nthreads)
{
    if (check_args(M, N, K, group_size, bits))
        return 1;
    for (int64_t i = 0; i < count; ++i)
        if (idx_m[i] < 0 || idx_m[i] >= M || idx_n[i] < 0 || idx_n[i] >= N)
            return 1;
    job_t j = {x, w_packed, scales, biases, M, N, K, group_size, bits, idx_m, idx_n, count,
               y_exact, y_bf16, 0, 0};
    return run_jobs(&j, nthreads, sampled_worker);
}

/* ---- quantization (test-data utility) --------------------------------- */

/* Min-max affine quantization of float weights w[N,K].  The pages give no
 * procedure; the plainest reading is used: per group, scale = (max-min) /
 * (2^bits - 1) and bias = min, both rounded to bf16; then
 * q = clamp(rint((w - bias) / scale), 0, 2^bits - 1) with the ROUNDED scale
 * and bias (ties to even).  A constant group gets scale 0 and q = 0. */
int aqo_quantize(const float *w, int64_t N, int64_t K, int group_size, int bits,
                 uint32_t *w_packed, uint16_t *scales, uint16_t *biases)
{
    if (check_args(1, N, K, group_size, bits))
        return 1;
    int64_t G = K / group_size;
    int qmax = (1 << bits) - 1;
    uint8_t *codes = (uint8_t *)malloc((size_t)(N * K));
    if (!codes)
        return 2;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < G; ++g) {
            const float *wg = w + n * K + g * group_size;
            double mn = wg[0], mx = wg[0];
            for (int i = 1; i < group_size; ++i) {
                if (wg[i] < mn)
                    mn = wg[i];
                if (wg[i] > mx)
                    mx = wg[i];
            }
            uint16_t s16 = aqo_double_to_bf16((mx - mn) / (double)qmax);
            uint16_t b16 = aqo_double_to_bf16(mn);
            scales[n * G + g] = s16;
            biases[n * G + g] = b16;
            double s = aqo_bf16_to_double(s16), b = aqo_bf16_to_double(b16);
            for (int i = 0; i < group_size; ++i) {
                double q = 0.0;
                if (s != 0.0) {
                    q = rint(((double)wg[i] - b) / s);
                    if (q < 0.0)
                        q = 0.0;
                    if (q > (double)qmax)
                        q = (double)qmax;
                }
                codes[n * K + g * group_size + i] = (uint8_t)q;
            }
        }
    int rc = aqo_pack(codes, N, K, bits, w_packed);
    free(codes);
    return rc;
}
