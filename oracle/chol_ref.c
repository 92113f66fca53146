/*
 * CPU ORACLE for batched single-precision Cholesky (SPOTRF, uplo = 'L' and 'U').
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file: only the tests, the package's smoke check and the benchmark's CPU
 * baseline leg do. It shares no code, header or table with the CUDA library.
 *
 * What it computes. For a symmetric positive definite A there is exactly one
 * lower-triangular L with a positive diagonal and A = L L^T, so the oracle is
 * that definition written out in the Cholesky-Crout ("dot product", column by
 * column, left-looking) order, in IEEE double with every operation rounded on
 * its own (the build passes -ffp-contract=off):
 *
 *   for j = 0 .. n-1
 *     d    = a_jj - sum_{k<j} l_jk^2                (summed left to right)
 *     if !(d > 0): info = j + 1, stop               (a NaN pivot fails too)
 *     l_jj = sqrt(d)
 *     for i = j+1 .. n-1
 *       l_ij = (a_ij - sum_{k<j} l_ik l_jk) / l_jj
 *
 * This is the recurrence stated in the comments of the chol_reg / chol_diag
 * kernels of "kernelbot-cholesky-930185" (the right-looking form there
 * computes the same numbers in another order) and the definition LAPACK's
 * unblocked potf2 implements ("BatchLAS perf_gemm", paragraph on TRSM
 * division and the POTRF reciprocal). info follows the statement of batched
 * SPOTRF: the 1-based index of the first pivot that is not positive, else 0.
 *
 * Only the lower triangle of the fp32 input is read, each entry converted
 * exactly to double. After a failure at pivot k only the leading (k-1)x(k-1)
 * block of L is defined; the oracle leaves the rest of L at zero.
 *
 * uplo = 'U' is the other half of LAPACK's potf2: A = U^T U with U upper
 * triangular, positive diagonal, only the upper triangle of A read. Written
 * out row by row of U in the same dot-product order:
 *
 *   for j = 0 .. n-1
 *     d    = a_jj - sum_{k<j} u_kj^2
 *     if !(d > 0): info = j + 1, stop
 *     u_jj = sqrt(d)
 *     for i = j+1 .. n-1
 *       u_ji = (a_ji - sum_{k<j} u_kj u_ki) / u_jj
 *
 * (U is the transpose of the lower factor of the same symmetric matrix, and
 * the sums run in the same order, so the two agree bit for bit.)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Factor one matrix. A is fp32 column-major with leading dimension lda (only
 * its lower triangle is read); L receives the double factor, column-major with
 * leading dimension ldl, strict upper triangle zero. Returns info. */
int oracle_potrf_one(const float *A, int n, int lda, double *L, int ldl)
{
    for (int j = 0; j < n; ++j)
        for (int i = 0; i < n; ++i)
            L[i + (int64_t)j * ldl] = 0.0;

    for (int j = 0; j < n; ++j) {
        double d = (double)A[j + (int64_t)j * lda];
        for (int k = 0; k < j; ++k) {
            const double ljk = L[j + (int64_t)k * ldl];
            d -= ljk * ljk;
        }
        if (!(d > 0.0))
            return j + 1;
        const double ljj = sqrt(d);
        L[j + (int64_t)j * ldl] = ljj;
        for (int i = j + 1; i < n; ++i) {
            double s = (double)A[i + (int64_t)j * lda];
            for (int k = 0; k < j; ++k)
                s -= L[i + (int64_t)k * ldl] * L[j + (int64_t)k * ldl];
            L[i + (int64_t)j * ldl] = s / ljj;
        }
    }
    return 0;
}

/* Factor one matrix, uplo = 'U'. A is fp32 column-major with leading
 * dimension lda (only its upper triangle, a_ij with i <= j at A[i + j*lda], is
 * read); U receives the double factor, column-major with leading dimension
 * ldu, strict lower triangle zero. Returns info. */
int oracle_potrf_upper_one(const float *A, int n, int lda, double *U, int ldu)
{
    for (int j = 0; j < n; ++j)
        for (int i = 0; i < n; ++i)
            U[i + (int64_t)j * ldu] = 0.0;

    for (int j = 0; j < n; ++j) {
        double d = (double)A[j + (int64_t)j * lda];
        for (int k = 0; k < j; ++k) {
            const double ukj = U[k + (int64_t)j * ldu];
            d -= ukj * ukj;
        }
        if (!(d > 0.0))
            return j + 1;
        const double ujj = sqrt(d);
        U[j + (int64_t)j * ldu] = ujj;
        for (int i = j + 1; i < n; ++i) {
            double s = (double)A[j + (int64_t)i * lda];
            for (int k = 0; k < j; ++k)
                s -= U[k + (int64_t)j * ldu] * U[k + (int64_t)i * ldu];
            U[j + (int64_t)i * ldu] = s / ujj;
        }
    }
    return 0;
}

typedef struct {
    const float *A;
    int n, lda;
    int64_t strideA;
    double *L;
    int64_t strideL;
    int *info;
    int upper;
    int b0, b1;
} oracle_job;

static void *oracle_worker(void *p)
{
    const oracle_job *job = (const oracle_job *)p;
    for (int b = job->b0; b < job->b1; ++b)
        job->info[b] = (job->upper ? oracle_potrf_upper_one : oracle_potrf_one)(
            job->A + (int64_t)b * job->strideA, job->n, job->lda,
            job->L + (int64_t)b * job->strideL, job->n);
    return NULL;
}

/* Factor a strided batch: matrix b is at A + b*strideA, its factor goes to
 * L + b*strideL (n x n, leading dimension n), info[b] receives its info.
 * uplo 'U' or 'u' factors A = U^T U from the upper triangles, anything else
 * A = L L^T from the lower. Work is split into contiguous slices over nthreads
 * POSIX threads (<= 0: one thread). Returns the number of threads used. */
int oracle_potrf_batched_uplo(char uplo, const float *A, int n, int lda, int64_t strideA,
                              int batch, double *L, int64_t strideL, int *info, int nthreads)
{
    if (batch <= 0)
        return 0;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > batch)
        nthreads = batch;
    oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    char *running = (char *)calloc((size_t)nthreads, 1);
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        oracle_job *j = &jobs[t];
        j->A = A; j->n = n; j->lda = lda; j->strideA = strideA;
        j->L = L; j->strideL = strideL; j->info = info;
        j->upper = (uplo == 'U' || uplo == 'u');
        j->b0 = (int)((int64_t)batch * t / nthreads);
        j->b1 = (int)((int64_t)batch * (t + 1) / nthreads);
        if (t == 0)
            continue;
        if (pthread_create(&tids[t], NULL, oracle_worker, j) == 0) {
            running[t] = 1;
            ++started;
        } else
            oracle_worker(j);  /* no thread: do the slice here */
    }
    oracle_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (running[t])
            pthread_join(tids[t], NULL);
    free(jobs);
    free(tids);
    free(running);
    return started + 1;
}

int oracle_potrf_batched(const float *A, int n, int lda, int64_t strideA, int batch,
                         double *L, int64_t strideL, int *info, int nthreads)
{
    return oracle_potrf_batched_uplo('L', A, n, lda, strideA, batch, L, strideL, info,
                                     nthreads);
}
