/*
 * CPU ORACLE for batched complex Cholesky (CPOTRF for single-precision and
 * ZPOTRF for double-precision complex input, uplo = 'L' and 'U'): for a
 * Hermitian positive definite A, A = L L^H with L lower
 * triangular and a real positive diagonal (uplo 'U': A = U^H U, U = L^H).
 * The definition written out in the Cholesky-Crout order, in double complex
 * with every operation rounded on its own (-ffp-contract=off):
 *
 *   d    = re(a_jj) - sum_{k<j} |l_jk|^2          (the diagonal's imaginary
 *                                                   part is not read, as LAPACK)
 *   !(d > 0): info = j + 1, stop
 *   l_jj = sqrt(d)
 *   l_ij = (a_ij - sum_{k<j} l_ik conj(l_jk)) / l_jj        (i > j)
 *
 * Input: interleaved complex (re, im) of floats (CPOTRF) or doubles (ZPOTRF),
 * column-major, leading dimension lda in complex elements, each part
 * converted exactly to double; only the lower (upper) triangle is read. TEST INFRASTRUCTURE ONLY, like chol_ref.c: nothing on
 * the product path links, loads or calls it. "BatchLAS perf_blackwell" lists
 * the complex types among its batched potrf types (its potrf type columns).
 */
#include <complex.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

/* element idx of the input: dbl = 0 interleaved floats, 1 interleaved doubles */
static double complex ld_c(const void *A, int dbl, int64_t idx)
{
    if (dbl)
        return ((const double *)A)[2 * idx] + ((const double *)A)[2 * idx + 1] * I;
    return (double)((const float *)A)[2 * idx] + (double)((const float *)A)[2 * idx + 1] * I;
}

/* Lower: a_ij (i >= j) at A[i + j*lda]; L: n x n double complex, leading
 * dimension ldl, strict upper zero. Returns info. */
static int potrf_lower(const void *A, int dbl, int n, int lda, double complex *L, int ldl)
{
    for (int j = 0; j < n; ++j)
        for (int i = 0; i < n; ++i)
            L[i + (int64_t)j * ldl] = 0.0;
    for (int j = 0; j < n; ++j) {
        double d = creal(ld_c(A, dbl, j + (int64_t)j * lda));
        for (int k = 0; k < j; ++k) {
            const double complex ljk = L[j + (int64_t)k * ldl];
            d -= creal(ljk) * creal(ljk) + cimag(ljk) * cimag(ljk);
        }
        if (!(d > 0.0))
            return j + 1;
        const double ljj = sqrt(d);
        L[j + (int64_t)j * ldl] = ljj;
        for (int i = j + 1; i < n; ++i) {
            double complex s = ld_c(A, dbl, i + (int64_t)j * lda);
            for (int k = 0; k < j; ++k)
                s -= L[i + (int64_t)k * ldl] * conj(L[j + (int64_t)k * ldl]);
            L[i + (int64_t)j * ldl] = s / ljj;
        }
    }
    return 0;
}

/* Upper: a_ij (i <= j) at A[i + j*lda]; U receives U = L^H, strict lower zero:
 * u_jj = sqrt(re(a_jj) - sum_{k<j} |u_kj|^2),
 * u_ji = (a_ji - sum_{k<j} conj(u_kj) u_ki) / u_jj   (i > j). */
static int potrf_upper(const void *A, int dbl, int n, int lda, double complex *U, int ldu)
{
    for (int j = 0; j < n; ++j)
        for (int i = 0; i < n; ++i)
            U[i + (int64_t)j * ldu] = 0.0;
    for (int j = 0; j < n; ++j) {
        double d = creal(ld_c(A, dbl, j + (int64_t)j * lda));
        for (int k = 0; k < j; ++k) {
            const double complex ukj = U[k + (int64_t)j * ldu];
            d -= creal(ukj) * creal(ukj) + cimag(ukj) * cimag(ukj);
        }
        if (!(d > 0.0))
            return j + 1;
        const double ujj = sqrt(d);
        U[j + (int64_t)j * ldu] = ujj;
        for (int i = j + 1; i < n; ++i) {
            double complex s = ld_c(A, dbl, j + (int64_t)i * lda);
            for (int k = 0; k < j; ++k)
                s -= conj(U[k + (int64_t)j * ldu]) * U[k + (int64_t)i * ldu];
            U[j + (int64_t)i * ldu] = s / ujj;
        }
    }
    return 0;
}

int oracle_cpotrf_one(const float *A, int n, int lda, double complex *L, int ldl)
{
    return potrf_lower(A, 0, n, lda, L, ldl);
}
int oracle_cpotrf_upper_one(const float *A, int n, int lda, double complex *U, int ldu)
{
    return potrf_upper(A, 0, n, lda, U, ldu);
}
int oracle_zpotrf_one(const double *A, int n, int lda, double complex *L, int ldl)
{
    return potrf_lower(A, 1, n, lda, L, ldl);
}
int oracle_zpotrf_upper_one(const double *A, int n, int lda, double complex *U, int ldu)
{
    return potrf_upper(A, 1, n, lda, U, ldu);
}

typedef struct {
    const void *A;
    int dbl;
    int n, lda;
    int64_t strideA;
    double complex *L;
    int64_t strideL;
    int *info;
    int upper;
    int b0, b1;
} cjob;

static void *cworker(void *p)
{
    const cjob *j = (const cjob *)p;
    const size_t esz = j->dbl ? 2 * sizeof(double) : 2 * sizeof(float);
    for (int b = j->b0; b < j->b1; ++b)
        j->info[b] = (j->upper ? potrf_upper : potrf_lower)(
            (const char *)j->A + (size_t)b * (size_t)j->strideA * esz, j->dbl, j->n, j->lda,
            j->L + (int64_t)b * j->strideL, j->n);
    return NULL;
}

/* A strided batch (strideA in complex elements) over nthreads threads; dbl
 * selects double-precision input. */
static int batched(char uplo, const void *A, int dbl, int n, int lda, int64_t strideA, int batch,
                   double complex *L, int64_t strideL, int *info, int nthreads)
{
    if (batch <= 0)
        return 0;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > batch)
        nthreads = batch;
    cjob *jobs = (cjob *)calloc((size_t)nthreads, sizeof(cjob));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    char *running = (char *)calloc((size_t)nthreads, 1);
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        cjob *j = &jobs[t];
        j->A = A; j->dbl = dbl; j->n = n; j->lda = lda; j->strideA = strideA;
        j->L = L; j->strideL = strideL; j->info = info;
        j->upper = (uplo == 'U' || uplo == 'u');
        j->b0 = (int)((int64_t)batch * t / nthreads);
        j->b1 = (int)((int64_t)batch * (t + 1) / nthreads);
        if (t == 0)
            continue;
        if (pthread_create(&tids[t], NULL, cworker, j) == 0) {
            running[t] = 1;
            ++started;
        } else
            cworker(j);
    }
    cworker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (running[t])
            pthread_join(tids[t], NULL);
    free(jobs);
    free(tids);
    free(running);
    return started + 1;
}

int oracle_cpotrf_batched_uplo(char uplo, const float *A, int n, int lda, int64_t strideA,
                               int batch, double complex *L, int64_t strideL, int *info,
                               int nthreads)
{
    return batched(uplo, A, 0, n, lda, strideA, batch, L, strideL, info, nthreads);
}

int oracle_zpotrf_batched_uplo(char uplo, const double *A, int n, int lda, int64_t strideA,
                               int batch, double complex *L, int64_t strideL, int *info,
                               int nthreads)
{
    return batched(uplo, A, 1, n, lda, strideA, batch, L, strideL, info, nthreads);
}
