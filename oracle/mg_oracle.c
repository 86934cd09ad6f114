/*
 * mg_oracle.c -- fp64 CPU oracle for Mirage's exp-normalised GQA kernel graph.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's CPU
 * baseline may load this library. The CUDA product path never links, calls or
 * falls back to it, and it shares no code, header or table with that path.
 *
 * What it computes (Mirage documentation, tutorials/group-query-attention,
 * "Define GQA Computation Graph"; the same graph opens section 1 of the blog
 * "Reading Mirage's muGraph search and backend generation through the GQA
 * example"):
 *
 *     A = matmul(Q, K)        Q (B,M,d), K (B,d,N)  ->  A (B,M,N)
 *     E = exp(A)
 *     S = reduction(E, 2)     sum over axis 2 (the N axis), kept as (B,M,1)
 *     D = div(E, S)           S broadcast along N
 *     O = matmul(D, V)        V (B,N,d)              ->  O (B,M,d)
 *
 * The graph has no max-subtraction and no 1/sqrt(d) scale, so neither is
 * applied here. Every step runs in IEEE double from the fp16 inputs, which are
 * widened exactly; exp is the C library's exp(double). The steps are taken in
 * the graph's order, one (b, m) row at a time, with no blocking or reordering
 * beyond that: the row is the unit over which reduction(E, 2) and div(E, S)
 * are defined.
 *
 * Layout: all tensors are contiguous row-major. Q[b][m][k], K[b][k][n],
 * V[b][n][c]; O[b][m][c] (double). fp16 values are passed as their raw
 * IEEE binary16 bit patterns (uint16_t).
 *
 * Threads: rows are independent; OpenMP spreads them over `nthreads` threads
 * (<= 0 means the OpenMP default). Results do not depend on the thread count.
 */

#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16 -> double, exactly: 1 sign bit, 5 exponent bits with bias
 * 15, 10 fraction bits. Subnormals are f * 2^-24; normals (1024 + f) *
 * 2^(e - 25); e == 31 encodes inf (f == 0) or NaN. */
static double half_bits_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25);
    return sign ? -v : v;
}

/* All 65536 binary16 bit patterns widened once; lookups are then exact and
 * cheap inside the row loops. */
static double g_half[65536];
static pthread_once_t g_half_once = PTHREAD_ONCE_INIT;

static void build_half_table(void)
{
    for (uint32_t h = 0; h < 65536u; ++h)
        g_half[h] = half_bits_to_double((uint16_t)h);
}

#define H(x) (g_half[(x)])

/* One output row O[b][m][:], following the graph step by step.
 * A, E are caller-provided scratch arrays of N doubles. */
static void oracle_row(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                       int64_t M, int64_t N, int64_t d, int64_t b, int64_t m,
                       double *A, double *E, double *out)
{
    const uint16_t *q = Q + (b * M + m) * d;   /* Q[b][m][:] */
    const uint16_t *Kb = K + b * d * N;        /* K[b][:][:] */
    const uint16_t *Vb = V + b * N * d;        /* V[b][:][:] */

    /* A[b,m,n] = sum_k Q[b,m,k] * K[b,k,n]   (matmul(Q, K)) */
    for (int64_t n = 0; n < N; ++n)
        A[n] = 0.0;
    for (int64_t k = 0; k < d; ++k) {
        const double qk = H(q[k]);
        const uint16_t *krow = Kb + k * N;
        for (int64_t n = 0; n < N; ++n)
            A[n] += qk * H(krow[n]);
    }

    /* E = exp(A) */
    for (int64_t n = 0; n < N; ++n)
        E[n] = exp(A[n]);

    /* S[b,m] = sum_n E[b,m,n]   (reduction(E, 2)) */
    double S = 0.0;
    for (int64_t n = 0; n < N; ++n)
        S += E[n];

    /* D[b,m,n] = E[b,m,n] / S[b,m]   (div(E, S)); stored over E */
    for (int64_t n = 0; n < N; ++n)
        E[n] = E[n] / S;

    /* O[b,m,c] = sum_n D[b,m,n] * V[b,n,c]   (matmul(D, V)) */
    for (int64_t c = 0; c < d; ++c)
        out[c] = 0.0;
    for (int64_t n = 0; n < N; ++n) {
        const double w = E[n];
        const uint16_t *vrow = Vb + n * d;
        for (int64_t c = 0; c < d; ++c)
            out[c] += w * H(vrow[c]);
    }
}

static int bad_shape(int64_t B, int64_t M, int64_t N, int64_t d)
{
    return B <= 0 || M <= 0 || N <= 0 || d <= 0;
}

/* Rows listed in `rows` (flat indices r = b*M + m, each in [0, B*M)) into
 * O[i][:] for i in [0, nrows). Returns 0 on success, -1 on a bad argument,
 * -2 when scratch memory cannot be had. */
int mg_oracle_attention_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                             int64_t B, int64_t M, int64_t N, int64_t d,
                             const int64_t *rows, int64_t nrows, int nthreads,
                             double *O)
{
    if (!Q || !K || !V || !O || !rows || nrows < 0 || bad_shape(B, M, N, d))
        return -1;
    for (int64_t i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= B * M)
            return -1;
    pthread_once(&g_half_once, build_half_table);
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#else
    nthreads = 1;
#endif
    int failed = 0;
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
    {
        double *A = (double *)malloc((size_t)N * sizeof(double));
        double *E = (double *)malloc((size_t)N * sizeof(double));
        if (!A || !E) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t i = 0; i < nrows; ++i) {
                const int64_t b = rows[i] / M;
                const int64_t m = rows[i] % M;
                oracle_row(Q, K, V, M, N, d, b, m, A, E, O + i * d);
            }
        }
        free(A);
        free(E);
    }
    return failed ? -2 : 0;
}

/* The whole output O (B, M, d) in double. Same return codes as above. */
int mg_oracle_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                        int64_t B, int64_t M, int64_t N, int64_t d, int nthreads,
                        double *O)
{
    if (!Q || !K || !V || !O || bad_shape(B, M, N, d))
        return -1;
    const int64_t nrows = B * M;
    int64_t *rows = (int64_t *)malloc((size_t)nrows * sizeof(int64_t));
    if (!rows)
        return -2;
    for (int64_t r = 0; r < nrows; ++r)
        rows[r] = r;
    const int rc = mg_oracle_attention_rows(Q, K, V, B, M, N, d, rows, nrows, nthreads, O);
    free(rows);
    return rc;
}

/* ------------------------------------------------------------------------
 * QK-norm attention (Mirage documentation, tutorials/attention-with-kv-norm,
 * "Implement QK Normalization and Optimize Attention Kernel in Python"):
 *
 *     Q = rms_norm(Q); K = rms_norm(K); then the graph above.
 *
 * rms_norm takes no weight in that graph. Reading: it normalises each query
 * row and each key vector over the head dimension d (for K, stored (B,d,N),
 * that is over axis 1), x / sqrt(mean(x^2) + eps), computed here in double
 * from the widened fp16 inputs and used unrounded.
 * ------------------------------------------------------------------------ */

/* One output row of QK-norm attention. A, E: scratch of N doubles; kn: scratch
 * of d*N doubles for the normalised key vectors of batch b. */
static void oracle_row_qknorm(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                              int64_t M, int64_t N, int64_t d, double eps, int64_t b,
                              int64_t m, double *A, double *E, double *qn, double *kn,
                              double *out)
{
    const uint16_t *q = Q + (b * M + m) * d;
    const uint16_t *Kb = K + b * d * N;
    const uint16_t *Vb = V + b * N * d;

    /* Q = rms_norm(Q): this row over d */
    double ss = 0.0;
    for (int64_t k = 0; k < d; ++k)
        ss += H(q[k]) * H(q[k]);
    const double rq = 1.0 / sqrt(ss / (double)d + eps);
    for (int64_t k = 0; k < d; ++k)
        qn[k] = H(q[k]) * rq;

    /* K = rms_norm(K): every key vector K[b][:][n] over d */
    for (int64_t n = 0; n < N; ++n) {
        double sk = 0.0;
        for (int64_t k = 0; k < d; ++k)
            sk += H(Kb[k * N + n]) * H(Kb[k * N + n]);
        const double rk = 1.0 / sqrt(sk / (double)d + eps);
        for (int64_t k = 0; k < d; ++k)
            kn[k * N + n] = H(Kb[k * N + n]) * rk;
    }

    /* A = matmul(Q, K) */
    for (int64_t n = 0; n < N; ++n)
        A[n] = 0.0;
    for (int64_t k = 0; k < d; ++k)
        for (int64_t n = 0; n < N; ++n)
            A[n] += qn[k] * kn[k * N + n];

    /* E = exp(A); S = reduction(E, 2); D = div(E, S); O = matmul(D, V) */
    for (int64_t n = 0; n < N; ++n)
        E[n] = exp(A[n]);
    double S = 0.0;
    for (int64_t n = 0; n < N; ++n)
        S += E[n];
    for (int64_t n = 0; n < N; ++n)
        E[n] = E[n] / S;
    for (int64_t c = 0; c < d; ++c)
        out[c] = 0.0;
    for (int64_t n = 0; n < N; ++n) {
        const double w = E[n];
        const uint16_t *vrow = Vb + n * d;
        for (int64_t c = 0; c < d; ++c)
            out[c] += w * H(vrow[c]);
    }
}

/* QK-norm attention for the listed rows (as mg_oracle_attention_rows); eps >= 0. */
int mg_oracle_attention_qknorm_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                    int64_t B, int64_t M, int64_t N, int64_t d, double eps,
                                    const int64_t *rows, int64_t nrows, int nthreads, double *O)
{
    if (!Q || !K || !V || !O || !rows || nrows < 0 || bad_shape(B, M, N, d) || !(eps >= 0.0))
        return -1;
    for (int64_t i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= B * M)
            return -1;
    pthread_once(&g_half_once, build_half_table);
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#else
    nthreads = 1;
#endif
    int failed = 0;
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
    {
        double *A = (double *)malloc((size_t)N * sizeof(double));
        double *E = (double *)malloc((size_t)N * sizeof(double));
        double *qn = (double *)malloc((size_t)d * sizeof(double));
        double *kn = (double *)malloc((size_t)d * (size_t)N * sizeof(double));
        if (!A || !E || !qn || !kn) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t i = 0; i < nrows; ++i)
                oracle_row_qknorm(Q, K, V, M, N, d, eps, rows[i] / M, rows[i] % M, A, E, qn, kn,
                                  O + i * d);
        }
        free(A);
        free(E);
        free(qn);
        free(kn);
    }
    return failed ? -2 : 0;
}

/* Threads OpenMP would use by default (1 when built without OpenMP). */
int mg_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
