/*
 * gemm_oracle.c -- CPU oracle for the fp16 GEMM  D = A * B^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the entry point's smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or table with the CUDA
 * library; the two meet only through the seeded input arrays.
 *
 * What it computes (the plain definition, written out):
 *
 *   D[m][n] = fp16_RNE( sum_{k<K} f64(A[m][k]) * f64(B[n][k]) )
 *
 *   - "GEMM I -- the tiled baseline", section "The problem we are solving":
 *     operands are fp16, the contraction runs at higher precision and the
 *     result is cast back to fp16 only at writeback; B is stored N x K
 *     row-major, so a row of B is a column of B^T.
 *   - same page, Step 1 pseudocode (writeback): the accumulator is rounded
 *     once, at the end.
 *   - "TIRx GEMM detailed technical notes", V8 "Operand Partition": the
 *     operation is D = A B^T, rows of the stored B become output columns.
 *
 * The pages accumulate in fp32; the oracle accumulates in fp64, which for
 * fp16 inputs is the exact sum for all practical purposes: every product of
 * two fp16 values has at most 22 significant bits and is exact in a double,
 * so the only rounding before the final cast is the fp64 running sum.
 *
 * The fp16 codec below is written from the IEEE 754 binary16 definition
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits; exponent 0 is
 * zero/subnormal with quantum 2^-24; exponent 31 is Inf/NaN).  The encoder
 * rounds a double straight to binary16, ties to even, with no float step in
 * between, so there is no double rounding.
 *
 * Built with -ffp-contract=off so that no multiply-add is fused on any host.
 * The ORACLE_MUTANT macro exists only so that the pin tests can prove they
 * catch a planted mistake; the shipped build never defines it.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ---------------------------------------------------------------- codec -- */

double oracle_f16_to_f64(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);                 /* zero or subnormal */
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;                    /* Inf or NaN        */
    } else {
        mag = ldexp((double)(1024 + frac), expo - 25);  /* normal            */
    }
    return sign ? -mag : mag;
}

uint16_t oracle_f64_to_f16(double x)
{
    if (isnan(x)) {
        return (uint16_t)(signbit(x) ? 0xfe00 : 0x7e00);
    }
    const uint16_t sign = signbit(x) ? 0x8000 : 0x0000;
    const double a = fabs(x);
    /* 65504 is the largest finite value; its fraction is odd, so the tie at
     * 65520 rounds up to 65536, which is out of range: Inf. */
    if (a >= 65520.0) {
        return (uint16_t)(sign | 0x7c00);
    }
    if (a == 0.0) {
        return sign;
    }
    int e2;
    (void)frexp(a, &e2);          /* a = f * 2^e2 with f in [0.5, 1)         */
    const int e = e2 - 1;         /* 2^e <= a < 2^(e+1)                      */
    const int subnormal = (e < -14);
    const int qexp = subnormal ? -24 : (e - 10);       /* log2 of the quantum  */
    const double n = ldexp(a, -qexp);                  /* exact: power-of-2 scale */
    const double fl = floor(n);
    const double rem = n - fl;                          /* exact               */
    double r = fl;
#if ORACLE_MUTANT == 3
    /* planted mistake: truncation instead of round-to-nearest-even */
    (void)rem;
#elif ORACLE_MUTANT == 4
    /* planted mistake: ties away from zero */
    if (rem >= 0.5) r = fl + 1.0;
#else
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) {
        r = fl + 1.0;
    }
#endif
    uint32_t bits;
    if (subnormal) {
        /* r in [0, 1024]; 1024 is the smallest normal, 0x0400, which the
         * same formula produces. */
        bits = (uint32_t)r;
    } else {
        /* r in [1024, 2048]; 2048 carries into the next binade, which the
         * same formula produces (and 0x7c00 = Inf past 65504). */
        bits = ((uint32_t)(e + 15) << 10) + ((uint32_t)r - 1024u);
    }
    return (uint16_t)(sign | bits);
}

void oracle_f16_to_f64_array(const uint16_t *src, double *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = oracle_f16_to_f64(src[i]);
}

void oracle_f64_to_f16_array(const double *src, uint16_t *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = oracle_f64_to_f16(src[i]);
}

/* ------------------------------------------------------ one dot product -- */

/* sum_{k<K} a[k] * b[k] in fp64, k ascending. */
static double dot_f64(const double *a, const double *b, int64_t K)
{
    double acc = 0.0;
#if ORACLE_MUTANT == 1
    /* planted mistake: the last term of the contraction is dropped */
    for (int64_t k = 0; k + 1 < K; ++k) acc += a[k] * b[k];
#elif ORACLE_MUTANT == 5
    /* planted mistake: fp32 running sum */
    float facc = 0.0f;
    for (int64_t k = 0; k < K; ++k) facc += (float)(a[k] * b[k]);
    acc = (double)facc;
#else
    for (int64_t k = 0; k < K; ++k) acc += a[k] * b[k];
#endif
    return acc;
}

/* ---------------------------------------------------------- full GEMM -- */

typedef struct {
    const double *Af;    /* M x K, decoded                                   */
    const double *Bf;    /* N x K, decoded (or K x N for mutant 2)           */
    uint16_t *D;         /* M x N                                            */
    double *Dacc;        /* M x N fp64 sums before rounding, may be NULL     */
    int64_t M, N, K;
    int64_t m_begin, m_end;
} gemm_job;

static void *gemm_rows(void *arg)
{
    const gemm_job *j = (const gemm_job *)arg;
    for (int64_t m = j->m_begin; m < j->m_end; ++m) {
        const double *a = j->Af + m * j->K;
        for (int64_t n = 0; n < j->N; ++n) {
            double acc;
#if ORACLE_MUTANT == 2
            /* planted mistake: B read as if it were stored K x N */
            acc = 0.0;
            for (int64_t k = 0; k < j->K; ++k) acc += a[k] * j->Bf[k * j->N + n];
#else
            acc = dot_f64(a, j->Bf + n * j->K, j->K);
#endif
            if (j->Dacc) j->Dacc[m * j->N + n] = acc;
            j->D[m * j->N + n] = oracle_f64_to_f16(acc);
        }
    }
    return NULL;
}

static int run_threads(void *(*fn)(void *), void *jobs, size_t job_size, int nthreads)
{
    if (nthreads <= 1) {
        fn(jobs);
        return 0;
    }
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!tid) return -1;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, fn, (char *)jobs + (size_t)t * job_size) != 0) break;
        ++started;
    }
    /* run whatever could not be started on this thread */
    for (int t = started; t < nthreads; ++t) fn((char *)jobs + (size_t)t * job_size);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    free(tid);
    return 0;
}

/*
 * D (M x N, fp16 bits) = RNE(A (M x K) * B (N x K)^T), all row-major.
 * Dacc, if not NULL, receives the fp64 sums before the final rounding.
 * threads <= 0 means 1.  Returns 0, or -1 on bad arguments / no memory.
 */
int oracle_gemm_f16_nt(const uint16_t *A, const uint16_t *B, uint16_t *D, double *Dacc,
                       int64_t M, int64_t N, int64_t K, int threads)
{
    if (M < 0 || N < 0 || K < 0 || (M * N > 0 && (!A || !B || !D))) return -1;
    if (M == 0 || N == 0) return 0;
    double *Af = (double *)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    double *Bf = (double *)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!Af || !Bf) {
        free(Af);
        free(Bf);
        return -1;
    }
    oracle_f16_to_f64_array(A, Af, M * K);
#if ORACLE_MUTANT == 2
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) Bf[k * N + n] = oracle_f16_to_f64(B[k * N + n]);
#else
    oracle_f16_to_f64_array(B, Bf, N * K);
#endif
    int nt = threads > 0 ? threads : 1;
    if (nt > M) nt = (int)M;
    gemm_job *jobs = (gemm_job *)calloc((size_t)nt, sizeof(gemm_job));
    if (!jobs) {
        free(Af);
        free(Bf);
        return -1;
    }
    for (int t = 0; t < nt; ++t) {
        jobs[t].Af = Af;
        jobs[t].Bf = Bf;
        jobs[t].D = D;
        jobs[t].Dacc = Dacc;
        jobs[t].M = M;
        jobs[t].N = N;
        jobs[t].K = K;
        jobs[t].m_begin = M * t / nt;
        jobs[t].m_end = M * (t + 1) / nt;
    }
    int rc = run_threads(gemm_rows, jobs, sizeof(gemm_job), nt);
    free(jobs);
    free(Af);
    free(Bf);
    return rc;
}

/* ------------------------------------------------------ sampled points -- */

typedef struct {
    const uint16_t *A, *B;
    int64_t M, N, K;
    const int64_t *rows, *cols;
    uint16_t *Dout;
    double *acc_out;
    int64_t begin, end;
    int status;
} point_job;

static void *gemm_points(void *arg)
{
    point_job *j = (point_job *)arg;
    double *a = (double *)malloc(sizeof(double) * (size_t)(j->K > 0 ? j->K : 1));
    double *b = (double *)malloc(sizeof(double) * (size_t)(j->K > 0 ? j->K : 1));
    if (!a || !b) {
        j->status = -1;
        free(a);
        free(b);
        return NULL;
    }
    for (int64_t i = j->begin; i < j->end; ++i) {
        const int64_t m = j->rows[i], n = j->cols[i];
        if (m < 0 || m >= j->M || n < 0 || n >= j->N) {
            j->status = -1;
            continue;
        }
        oracle_f16_to_f64_array(j->A + m * j->K, a, j->K);
        oracle_f16_to_f64_array(j->B + n * j->K, b, j->K);
        const double acc = dot_f64(a, b, j->K);
        if (j->acc_out) j->acc_out[i] = acc;
        j->Dout[i] = oracle_f64_to_f16(acc);
    }
    free(a);
    free(b);
    return NULL;
}

/*
 * The same definition at `count` chosen output points (rows[i], cols[i]):
 * Dout[i] = D[rows[i]][cols[i]], acc_out[i] (may be NULL) its fp64 sum.
 * Returns 0, or -1 on bad arguments (an index out of range) / no memory.
 */
int oracle_gemm_f16_nt_points(const uint16_t *A, const uint16_t *B, int64_t M, int64_t N, int64_t K,
                              const int64_t *rows, const int64_t *cols, int64_t count,
                              uint16_t *Dout, double *acc_out, int threads)
{
    if (M < 0 || N < 0 || K < 0 || count < 0) return -1;
    if (count == 0) return 0;
    if (!A || !B || !rows || !cols || !Dout) return -1;
    int nt = threads > 0 ? threads : 1;
    if (nt > count) nt = (int)count;
    point_job *jobs = (point_job *)calloc((size_t)nt, sizeof(point_job));
    if (!jobs) return -1;
    for (int t = 0; t < nt; ++t) {
        jobs[t].A = A;
        jobs[t].B = B;
        jobs[t].M = M;
        jobs[t].N = N;
        jobs[t].K = K;
        jobs[t].rows = rows;
        jobs[t].cols = cols;
        jobs[t].Dout = Dout;
        jobs[t].acc_out = acc_out;
        jobs[t].begin = count * t / nt;
        jobs[t].end = count * (t + 1) / nt;
        jobs[t].status = 0;
    }
    int rc = run_threads(gemm_points, jobs, sizeof(point_job), nt);
    for (int t = 0; t < nt; ++t)
        if (jobs[t].status) rc = -1;
    free(jobs);
    return rc;
}
