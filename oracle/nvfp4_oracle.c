/*
 * nvfp4_oracle.c -- plain, slow CPU oracle for the grouped NVFP4 block-scaled GEMM.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg use this file. The CUDA library shares no code
 * with it, and neither includes the other.
 *
 * What it computes. For each group i, each m < M_i and each n < N_i:
 *
 *   C_i[m][n] = fp16_rne( sum_{k < K_i}  e2m1(A_i[m][k]) * e4m3(SFA_i[m][k/16])
 *                                      * e2m1(B_i[n][k]) * e4m3(SFB_i[n][k/16]) )
 *
 * Sources:
 *  - Page 2, submission 505431, python section, `custom_kernel_fallback`.
 *    It dequantises A and B, multiplies each element by the scale of its
 *    16-element block (`repeat_interleave(16)` in `apply_scale_factors`),
 *    computes C = A . B^T and casts the result to fp16.
 *  - Page 3, submission 444497, kernel header comment.
 *    C[i](M_i x N_i) = A[i](M_i x K_i) @ B[i](N_i x K_i)^T, with E2M1 data,
 *    E4M3FN scales and fp16 output.
 *
 * Precision. Products and sums are taken in IEEE double. The result is rounded
 * to fp16 once, with this file's own round-to-nearest-even.
 *
 * Exactness. With E2M1 magnitudes <= 6 (quantum 1/2) and E4M3 scales in
 * [2^-3, 2^1] (quantum 2^-6), each product is a multiple of 2^-14 of size
 * <= 144. A sum of at most 2^16 such products needs fewer than 53
 * significant bits, so the double sum is exact. The returned fp16 is then
 * the correctly rounded value of the exact result.
 *
 * Readings taken where the pages leave a step open:
 *  - Element 2j of a row is the low nibble of byte j, and element 2j+1 is the
 *    high nibble (page 2, python section, `dequantize_fp4`).
 *  - Scales are E4M3FN: no infinities, and 0x7F/0xFF are NaN. The sign bit is
 *    decoded even though the tensor-core scale type has none, so that misuse
 *    shows up in tests.
 *  - E2M1 code 8 is -0, which contributes nothing.
 *
 * Built with -ffp-contract=off, so no FMA merges a product into a sum and the
 * results are the same on x86-64 and aarch64.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t M, N, K;
    const uint8_t *A;   /* [M][K/2] packed E2M1 pairs                  */
    const uint8_t *B;   /* [N][K/2] packed E2M1 pairs                  */
    const uint8_t *SFA; /* [M][K/16] E4M3 scale bytes, row-major       */
    const uint8_t *SFB; /* [N][K/16] E4M3 scale bytes, row-major       */
    uint16_t *C;        /* out: [M][N] fp16 bit patterns               */
    double *S;          /* out, may be NULL: [M][N] sum_k |a*sa*b*sb|  */
} OracleProblem;

/* ---- element decoders ---------------------------------------------------- */

/* E2M1 code -> value. The magnitudes come from the 16-entry table on page 2
 * (python section, `_E2M1_LUT`): codes 0..7 give 0, .5, 1, 1.5, 2, 3, 4, 6, and
 * bit 3 is the sign. */
double oracle_e2m1(unsigned code)
{
    static const double magnitude[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double v = magnitude[code & 7u];
    return (code & 8u) ? -v : v;
}

/* E4M3 (FN variant) byte -> value, decoded from its bit fields:
 * sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0.
 * exponent 0 is subnormal: m/8 * 2^-6. exponent 15 with mantissa 7 is NaN.
 * Every other code is normal: (1 + m/8) * 2^(e-7). */
double oracle_e4m3(unsigned byte)
{
    unsigned s = (byte >> 7) & 1u, e = (byte >> 3) & 15u, m = byte & 7u;
    double v;
    if (e == 15u && m == 7u)
        return NAN;
    if (e == 0u)
        v = ldexp((double)m, -9);               /* m/8 * 2^-6 */
    else
        v = ldexp((double)(8u + m), (int)e - 10); /* (8+m)/8 * 2^(e-7) */
    return s ? -v : v;
}

/* ---- double -> fp16, round to nearest, ties to even ---------------------- */

/* Round a non-negative double to the nearest integer, with ties going to the
 * even integer. The argument is below 2^12 here, so it is exact in double and
 * so are floor and the difference. */
static double round_half_even(double q)
{
    double n = floor(q), frac = q - n;
    if (frac > 0.5)
        return n + 1.0;
    if (frac < 0.5)
        return n;
    return (fmod(n, 2.0) == 0.0) ? n : n + 1.0;
}

uint16_t oracle_fp16_rne(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x))
        return (uint16_t)(sign | 0x7E00u);
    double a = fabs(x);
    /* 65520 = 65504 + half a quantum: from here up, the value rounds to inf. */
    if (a >= 65520.0)
        return (uint16_t)(sign | 0x7C00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: quantum 2^-24; n = 1024 carries into the smallest normal */
        double n = round_half_even(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)n);
    }
    int e2;
    frexp(a, &e2);   /* a = f * 2^e2 with f in [0.5, 1) */
    int E = e2 - 1;  /* a in [2^E, 2^(E+1)), -14 <= E <= 15 */
    double n = round_half_even(ldexp(a, 10 - E)); /* in [1024, 2048] */
    if (n == 2048.0) {
        n = 1024.0;
        E += 1;
    }
    if (E > 15)
        return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(n - 1024.0));
}

/* ---- the grouped GEMM ---------------------------------------------------- */

static double element(const uint8_t *row, const uint8_t *sfrow, int k)
{
    unsigned byte = row[k >> 1];
    unsigned code = (k & 1) ? (byte >> 4) : (byte & 15u);
    return oracle_e2m1(code) * oracle_e4m3(sfrow[k >> 4]);
}

typedef struct {
    const OracleProblem *p;
    double *bdq;   /* dequantised B: [N][K] */
    int pass;      /* 0: dequantise B rows, 1: compute C rows */
    int tid, nthreads;
} Work;

static void *worker(void *arg)
{
    Work *w = (Work *)arg;
    const OracleProblem *p = w->p;
    const int K = p->K, kb = K / 2, ks = K / 16;
    if (w->pass == 0) {
        for (int n = w->tid; n < p->N; n += w->nthreads)
            for (int k = 0; k < K; ++k)
                w->bdq[(size_t)n * K + k] = element(p->B + (size_t)n * kb, p->SFB + (size_t)n * ks, k);
        return NULL;
    }
    double *arow = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    if (!arow)
        return (void *)1;
    for (int m = w->tid; m < p->M; m += w->nthreads) {
        for (int k = 0; k < K; ++k)
            arow[k] = element(p->A + (size_t)m * kb, p->SFA + (size_t)m * ks, k);
        for (int n = 0; n < p->N; ++n) {
            const double *brow = w->bdq + (size_t)n * K;
            double acc = 0.0, mag = 0.0;
            for (int k = 0; k < K; ++k) {
                double t = arow[k] * brow[k];
                acc += t;
                mag += fabs(t);
            }
            p->C[(size_t)m * p->N + n] = oracle_fp16_rne(acc);
            if (p->S)
                p->S[(size_t)m * p->N + n] = mag;
        }
    }
    free(arow);
    return NULL;
}

static int run_pass(const OracleProblem *p, double *bdq, int pass, int nthreads)
{
    pthread_t th[256];
    Work w[256];
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    int started = 0, rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        w[t].p = p;
        w[t].bdq = bdq;
        w[t].pass = pass;
        w[t].tid = t;
        w[t].nthreads = nthreads;
        if (pthread_create(&th[t], NULL, worker, &w[t]) != 0) {
            rc = -1;
            break;
        }
        ++started;
    }
    for (int t = 0; t < started; ++t) {
        void *ret = NULL;
        pthread_join(th[t], &ret);
        if (ret)
            rc = -1;
    }
    return rc;
}

/* Fills C (and S when non-NULL) of every group. Returns 0, or -1 on a bad
 * shape or an allocation failure. */
int oracle_grouped_gemm(int g, const OracleProblem *probs, int nthreads)
{
    if (g < 0 || (g > 0 && !probs))
        return -1;
    for (int i = 0; i < g; ++i) {
        const OracleProblem *p = &probs[i];
        if (p->M < 0 || p->N < 0 || p->K < 0 || p->K % 16 != 0)
            return -1;
        if (p->M == 0 || p->N == 0)
            continue;
        double *bdq = (double *)malloc(sizeof(double) * ((size_t)p->N * (size_t)p->K + 1));
        if (!bdq)
            return -1;
        int rc = run_pass(p, bdq, 0, nthreads);
        if (rc == 0)
            rc = run_pass(p, bdq, 1, nthreads);
        free(bdq);
        if (rc != 0)
            return rc;
    }
    return 0;
}

/* Computes only the listed outputs (m[i], n[i]) of one problem, one by one.
 * c[i] and s[i] receive the value and the magnitude sum (s may be NULL).
 * p->C and p->S are not used. */
int oracle_gemm_entries(const OracleProblem *p, int count, const int32_t *m, const int32_t *n,
                        uint16_t *c, double *s)
{
    if (!p || p->K < 0 || p->K % 16 != 0 || count < 0)
        return -1;
    const int K = p->K, kb = K / 2, ks = K / 16;
    for (int i = 0; i < count; ++i) {
        if (m[i] < 0 || m[i] >= p->M || n[i] < 0 || n[i] >= p->N)
            return -1;
        const uint8_t *ar = p->A + (size_t)m[i] * kb, *sar = p->SFA + (size_t)m[i] * ks;
        const uint8_t *br = p->B + (size_t)n[i] * kb, *sbr = p->SFB + (size_t)n[i] * ks;
        double acc = 0.0, mag = 0.0;
        for (int k = 0; k < K; ++k) {
            double t = element(ar, sar, k) * element(br, sbr, k);
            acc += t;
            mag += fabs(t);
        }
        c[i] = oracle_fp16_rne(acc);
        if (s)
            s[i] = mag;
    }
    return 0;
}

/* ---- the blocked ("128 x 4") scale layout -------------------------------- */

/* Page 4, submission 482006, `to_blocked_gpu`, gives the steps:
 *  1. Zero-pad the rows x cols scale matrix to R = 128*ceil(rows/128) rows and
 *     C = 4*ceil(cols/4) columns.
 *  2. Cut it into 128 x 4 blocks, row-block major with column blocks inner.
 *  3. Inside a block, write row r = 32*i + j, column c as byte j*16 + i*4 + c.
 * The same page's layout comment gives this block as the "atom" with shape
 * ((32,4),(16,4)) and strides ((16,4),(0,1)).
 *
 * Output byte count: R * C. The loops run in output order. */
size_t oracle_blocked_scale_bytes(int rows, int cols)
{
    if (rows <= 0 || cols <= 0)
        return 0;
    size_t R = (size_t)((rows + 127) / 128) * 128, C = (size_t)((cols + 3) / 4) * 4;
    return R * C;
}

int oracle_blocked_scales(const uint8_t *sf, int rows, int cols, uint8_t *out)
{
    if (rows < 0 || cols < 0)
        return -1;
    int nrb = (rows + 127) / 128, ncb = (cols + 3) / 4;
    size_t o = 0;
    for (int rb = 0; rb < nrb; ++rb)
        for (int cb = 0; cb < ncb; ++cb)
            for (int j = 0; j < 32; ++j)
                for (int i = 0; i < 4; ++i)
                    for (int c4 = 0; c4 < 4; ++c4) {
                        int r = rb * 128 + i * 32 + j, c = cb * 4 + c4;
                        out[o++] = (r < rows && c < cols) ? sf[(size_t)r * cols + c] : 0;
                    }
    return 0;
}
