/*
 * CPU ORACLE for batched double-precision Cholesky (DPOTRF, uplo = 'L' and
 * 'U'): the definition chol_ref.c writes out for the single-precision input,
 * here for a double-precision input, in IEEE double with every operation
 * rounded on its own (-ffp-contract=off), in the same Cholesky-Crout order:
 *
 *   lower:  d = a_jj - sum_{k<j} l_jk^2;  !(d > 0) -> info = j + 1, stop;
 *           l_jj = sqrt(d);  l_ij = (a_ij - sum_{k<j} l_ik l_jk) / l_jj  (i > j)
 *   upper:  the same with u_kj = l_jk, reading and writing the upper triangle.
 *
 * TEST INFRASTRUCTURE ONLY, like chol_ref.c: nothing on the product path
 * links, loads or calls it, and it shares no code with the CUDA library.
 * "BatchLAS perf_blackwell" lists the double type among the batched potrf
 * types (its potrf rows and type columns).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

/* Lower: only a_ij with i >= j is read (column-major, leading dimension lda);
 * L (n x n, leading dimension ldl) receives the factor, strict upper zero. */
int oracle_dpotrf_one(const double *A, int n, int lda, double *L, int ldl)
{
    for (int j = 0; j < n; ++j)
        for (int i = 0; i < n; ++i)
            L[i + (int64_t)j * ldl] = 0.0;
    for (int j = 0; j < n; ++j) {
        double d = A[j + (int64_t)j * lda];
        for (int k = 0; k < j; ++k) {
            const double ljk = L[j + (int64_t)k * ldl];
            d -= ljk * ljk;
        }
        if (!(d > 0.0))
            return j + 1;
        const double ljj = sqrt(d);
        L[j + (int64_t)j * ldl] = ljj;
        for (int i = j + 1; i < n; ++i) {
            double s = A[i + (int64_t)j * lda];
            for (int k = 0; k < j; ++k)
                s -= L[i + (int64_t)k * ldl] * L[j + (int64_t)k * ldl];
            L[i + (int64_t)j * ldl] = s / ljj;
        }
    }
    return 0;
}

/* Upper: only a_ij with i <= j is read; U receives the factor, strict lower zero. */
int oracle_dpotrf_upper_one(const double *A, int n, int lda, double *U, int ldu)
{
    for (int j = 0; j < n; ++j)
        for (int i = 0; i < n; ++i)
            U[i + (int64_t)j * ldu] = 0.0;
    for (int j = 0; j < n; ++j) {
        double d = A[j + (int64_t)j * lda];
        for (int k = 0; k < j; ++k) {
            const double ukj = U[k + (int64_t)j * ldu];
            d -= ukj * ukj;
        }
        if (!(d > 0.0))
            return j + 1;
        const double ujj = sqrt(d);
        U[j + (int64_t)j * ldu] = ujj;
        for (int i = j + 1; i < n; ++i) {
            double s = A[j + (int64_t)i * lda];
            for (int k = 0; k < j; ++k)
                s -= U[k + (int64_t)j * ldu] * U[k + (int64_t)i * ldu];
            U[j + (int64_t)i * ldu] = s / ujj;
        }
    }
    return 0;
}

typedef struct {
    const double *A;
    int n, lda;
    int64_t strideA;
    double *L;
    int64_t strideL;
    int *info;
    int upper;
    int b0, b1;
} djob;

static void *dworker(void *p)
{
    const djob *j = (const djob *)p;
    for (int b = j->b0; b < j->b1; ++b)
        j->info[b] = (j->upper ? oracle_dpotrf_upper_one : oracle_dpotrf_one)(
            j->A + (int64_t)b * j->strideA, j->n, j->lda, j->L + (int64_t)b * j->strideL, j->n);
    return NULL;
}

/* A strided batch over nthreads POSIX threads; uplo 'U'/'u' upper, else lower.
 * Returns the number of threads used. */
int oracle_dpotrf_batched_uplo(char uplo, const double *A, int n, int lda, int64_t strideA,
                               int batch, double *L, int64_t strideL, int *info, int nthreads)
{
    if (batch <= 0)
        return 0;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > batch)
        nthreads = batch;
    djob *jobs = (djob *)calloc((size_t)nthreads, sizeof(djob));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    char *running = (char *)calloc((size_t)nthreads, 1);
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        djob *j = &jobs[t];
        j->A = A; j->n = n; j->lda = lda; j->strideA = strideA;
        j->L = L; j->strideL = strideL; j->info = info;
        j->upper = (uplo == 'U' || uplo == 'u');
        j->b0 = (int)((int64_t)batch * t / nthreads);
        j->b1 = (int)((int64_t)batch * (t + 1) / nthreads);
        if (t == 0)
            continue;
        if (pthread_create(&tids[t], NULL, dworker, j) == 0) {
            running[t] = 1;
            ++started;
        } else
            dworker(j);
    }
    dworker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (running[t])
            pthread_join(tids[t], NULL);
    free(jobs);
    free(tids);
    free(running);
    return started + 1;
}
