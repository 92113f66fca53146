/*
 * CPU ORACLE for batched single-precision SPOTRS (uplo = 'L' and 'U'): solve
 * A X = B for every matrix of a batch, given the Cholesky factor of A.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file: only the tests and the benchmark's CPU baseline leg do. It shares
 * no code, header or table with the CUDA library.
 *
 * What it computes. With A = L L^T, A X = B is the two triangular solves the
 * posv row of "BatchLAS perf_blackwell" composes (posv = potrf followed by
 * two TRSMs; "BatchLAS perf_trsm" fuses them for the tiny sizes): first
 * L Y = B, then L^T X = Y, each right-hand side column on its own, written
 * out as plain substitution in IEEE double with every operation rounded on
 * its own (the build passes -ffp-contract=off):
 *
 *   forward   for i = 0 .. n-1:    y_i = (b_i - sum_{k<i} l_ik y_k) / l_ii
 *   backward  for i = n-1 .. 0:    x_i = (y_i - sum_{k>i} l_ki x_k) / l_ii
 *
 * (sums left to right in k). Only the lower triangle of the fp32 factor is
 * read, each entry converted exactly to double; B is fp32, X is double.
 *
 * With uplo = 'U' the factor is U (A = U^T U, upper triangle read): first
 * U^T y = b, then U x = y:
 *
 *   forward   for i = 0 .. n-1:    y_i = (b_i - sum_{k<i} u_ki y_k) / u_ii
 *   backward  for i = n-1 .. 0:    x_i = (y_i - sum_{k>i} u_ik x_k) / u_ii
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

/* One matrix. L: fp32 column-major, leading dimension lda (lower triangle
 * read). B: fp32 n x nrhs column-major, leading dimension ldb. X: double
 * n x nrhs column-major, leading dimension ldx (X may not alias B). */
void oracle_potrs_one(const float *L, int n, int lda, const float *B, int nrhs, int ldb,
                      double *X, int ldx)
{
    for (int c = 0; c < nrhs; ++c) {
        const float *b = B + (int64_t)c * ldb;
        double *x = X + (int64_t)c * ldx;
        /* forward: L y = b (y kept in x) */
        for (int i = 0; i < n; ++i) {
            double s = (double)b[i];
            for (int k = 0; k < i; ++k)
                s -= (double)L[i + (int64_t)k * lda] * x[k];
            x[i] = s / (double)L[i + (int64_t)i * lda];
        }
        /* backward: L^T x = y */
        for (int i = n - 1; i >= 0; --i) {
            double s = x[i];
            for (int k = i + 1; k < n; ++k)
                s -= (double)L[k + (int64_t)i * lda] * x[k];
            x[i] = s / (double)L[i + (int64_t)i * lda];
        }
    }
}

/* One matrix, uplo = 'U'. U: fp32 column-major, leading dimension lda (upper
 * triangle read, u_ij with i <= j at U[i + j*lda]). B, X as above. */
void oracle_potrs_upper_one(const float *U, int n, int lda, const float *B, int nrhs, int ldb,
                            double *X, int ldx)
{
    for (int c = 0; c < nrhs; ++c) {
        const float *b = B + (int64_t)c * ldb;
        double *x = X + (int64_t)c * ldx;
        /* forward: U^T y = b */
        for (int i = 0; i < n; ++i) {
            double s = (double)b[i];
            for (int k = 0; k < i; ++k)
                s -= (double)U[k + (int64_t)i * lda] * x[k];
            x[i] = s / (double)U[i + (int64_t)i * lda];
        }
        /* backward: U x = y */
        for (int i = n - 1; i >= 0; --i) {
            double s = x[i];
            for (int k = i + 1; k < n; ++k)
                s -= (double)U[i + (int64_t)k * lda] * x[k];
            x[i] = s / (double)U[i + (int64_t)i * lda];
        }
    }
}

typedef struct {
    const float *L;
    int n, lda;
    int64_t strideA;
    const float *B;
    int nrhs, ldb;
    int64_t strideB;
    double *X;
    int64_t strideX;
    int upper;
    int b0, b1;
} potrs_job;

static void *potrs_worker(void *p)
{
    const potrs_job *j = (const potrs_job *)p;
    for (int b = j->b0; b < j->b1; ++b)
        (j->upper ? oracle_potrs_upper_one : oracle_potrs_one)(j->L + (int64_t)b * j->strideA, j->n, j->lda,
                         j->B + (int64_t)b * j->strideB, j->nrhs, j->ldb,
                         j->X + (int64_t)b * j->strideX, j->n);
    return NULL;
}

/* A strided batch: factor b at L + b*strideA, right-hand sides at
 * B + b*strideB, solution to X + b*strideX (n x nrhs, leading dimension n).
 * uplo 'U' or 'u': the factors are upper (A = U^T U), else lower.
 * Contiguous slices over nthreads POSIX threads; returns the threads used. */
int oracle_potrs_batched_uplo(char uplo, const float *L, int n, int lda, int64_t strideA,
                              const float *B, int nrhs, int ldb, int64_t strideB, int batch,
                              double *X, int64_t strideX, int nthreads)
{
    if (batch <= 0)
        return 0;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > batch)
        nthreads = batch;
    potrs_job *jobs = (potrs_job *)calloc((size_t)nthreads, sizeof(potrs_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    char *running = (char *)calloc((size_t)nthreads, 1);
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        potrs_job *j = &jobs[t];
        j->L = L; j->n = n; j->lda = lda; j->strideA = strideA;
        j->B = B; j->nrhs = nrhs; j->ldb = ldb; j->strideB = strideB;
        j->X = X; j->strideX = strideX;
        j->upper = (uplo == 'U' || uplo == 'u');
        j->b0 = (int)((int64_t)batch * t / nthreads);
        j->b1 = (int)((int64_t)batch * (t + 1) / nthreads);
        if (t == 0)
            continue;
        if (pthread_create(&tids[t], NULL, potrs_worker, j) == 0) {
            running[t] = 1;
            ++started;
        } else
            potrs_worker(j);
    }
    potrs_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (running[t])
            pthread_join(tids[t], NULL);
    free(jobs);
    free(tids);
    free(running);
    return started + 1;
}

int oracle_potrs_batched(const float *L, int n, int lda, int64_t strideA, const float *B,
                         int nrhs, int ldb, int64_t strideB, int batch, double *X,
                         int64_t strideX, int nthreads)
{
    return oracle_potrs_batched_uplo('L', L, n, lda, strideA, B, nrhs, ldb, strideB, batch, X,
                                     strideX, nthreads);
}
