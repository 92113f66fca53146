/*
 * bl_spotrf.h - batched single-precision Cholesky factorization (SPOTRF,
 * uplo = 'L' or 'U') and the solves with the factor (SPOTRS, SPOSV) for many
 * small independent matrices on one NVIDIA GB300 (sm_103a).
 *
 * The operation. For each b < batch, the symmetric positive definite matrix
 * A_b = A + b*strideA (column-major, element (i, j) at A_b[i + j*lda]) is
 * factored as A_b = L_b L_b^T with L_b lower triangular with a positive
 * diagonal, and L_b overwrites the lower triangle of A_b in place:
 *
 *     d_j  = a_jj - sum_{k<j} l_jk^2,   l_jj = sqrt(d_j),
 *     l_ij = (a_ij - sum_{k<j} l_ik l_jk) / l_jj          (i > j).
 *
 * This is the problem stated by the batched Cholesky leaderboard task of
 * "kernelbot-cholesky-930185" (its problem statement and the chol_reg /
 * chol_diag kernel comments; there row-major, a fresh output and a zeroed
 * upper triangle) and the per-matrix factor of "BatchLAS perf_blackwell"
 * (potrf rows of its routing table). Here the layout is the LAPACK one:
 * column-major, strided batch, lower triangle written in place, everything
 * else untouched.
 *
 * info[b] = 0 when every pivot d_j was > 0, else the 1-based index j+1 of the
 * first pivot with !(d_j > 0) (a NaN pivot fails; +Inf passes; a positive
 * pivot below FLT_MIN, a subnormal, is read as zero the way flush-to-zero
 * single precision reads it, and fails). After a
 * failure at k = info[b] only the leading (k-1) x (k-1) block of L_b is
 * defined; the rest of that matrix's lower triangle is unspecified.
 * info[b] = -1 reports an internal error: a bounded wait inside a
 * tensor-core kernel gave up (about a second) and matrix b's result is not
 * valid. It does not occur in normal operation.
 *
 * All arithmetic is IEEE single precision (contractions into FMA allowed; the
 * reciprocal square root of the pivot is the hardware approximation).
 */
#ifndef BL_SPOTRF_H
#define BL_SPOTRF_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Largest n the library factors (argument check -7 above it). */
#define BL_SPOTRF_MAX_N 4096

/* Route numbers of bl_spotrf_batched_ex and bl_spotrf_route. */
#define BL_ROUTE_AUTO 0
#define BL_ROUTE_WARP 1     /* K1: one warp (or a 16/8-lane group) per matrix, n <= 64 */
#define BL_ROUTE_CTA 2      /* one thread block per matrix, n <= 128: K2 (shared-memory
                               resident, bulk copies) for n <= 64 and the aligned orders
                               96 and 128, else a warp per 32 x 32 tile in registers */
#define BL_ROUTE_BLOCKED 3  /* K3: right-looking blocked, 128-wide panels: diagonal factor,
                               panel triangular solve, lower-only trailing update, any n
                               (forced: the right-looking order at any batch) */
#define BL_ROUTE_TMEM 4     /* K2t: one thread block per matrix, the matrix resident in tensor
                               memory, trailing updates on the tensor cores, n <= 128 */
#define BL_ROUTE_LEFT 5     /* K3's kernels in the left-looking order: per panel, its columns
                               updated by every earlier panel at once, then its diagonal
                               factor and panel solve; n > 128 (unaligned batches: K3) */

/*
 * bl_spotrf_batched - factor a strided batch in place.
 *
 *   A        device pointer to matrix 0 (float, column-major). Only the lower
 *            triangle (i >= j, i < n) of each matrix is read and written; the
 *            strict upper triangle, the rows n..lda-1 of every column and the
 *            memory between matrices are never read or written. Any alignment
 *            of 4 bytes is accepted; 16-byte alignment of A, lda and strideA
 *            lets the kernels use vector loads.
 *   n        order of every matrix (n >= 0).
 *   lda      leading dimension, lda >= max(1, n).
 *   strideA  distance in floats between A_b and A_{b+1}; strideA >= lda*n
 *            when batch > 1 (matrices may not overlap).
 *   batch    number of matrices (batch >= 0).
 *   info     device pointer to batch ints, written once per matrix (no
 *            pre-fill needed).
 *   stream   CUDA stream the work is enqueued on (0 = the legacy default).
 *
 * Ownership: the caller owns A and info (any device allocation, e.g. torch
 * tensors). The library allocates nothing, keeps no per-call state, does not
 * synchronize, and is reentrant and safe to call from several host threads
 * and streams at once. Work on one (A, info) is ordered by `stream`.
 *
 * Returns 0 when the work was enqueued; a negative value -i when argument i is
 * invalid (nothing is enqueued):
 *   -1 A == NULL while n > 0 and batch > 0     -2 n < 0
 *   -3 lda < max(1, n)                          -4 batch > 1 and strideA < lda*n
 *   -5 batch < 0                                -6 info == NULL while batch > 0
 *   -7 n > BL_SPOTRF_MAX_N
 * Arguments are checked in the order -2, -5, -3, -4, -1, -6, -7. A positive
 * value is the cudaError_t of a failed launch. Matrix-level failure (a matrix
 * that is not positive definite) is reported only through info.
 * Quick returns: batch == 0 enqueues nothing; n == 0 sets info[b] = 0 for all b.
 */
int bl_spotrf_batched(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                      cudaStream_t stream);

/*
 * bl_spotrf_batched_ex - as bl_spotrf_batched, with the kernel class forced
 * (route = BL_ROUTE_*; BL_ROUTE_AUTO selects like bl_spotrf_batched: by n, and
 * above n = 256 by batch between BL_ROUTE_BLOCKED and BL_ROUTE_LEFT, as
 * bl_spotrf_route reports).
 * Returns -8 when the forced route cannot factor this n (WARP: n > 64;
 * CTA or TMEM: n > 128; LEFT: n <= 128), after the checks above. For tests
 * and measurement.
 */
int bl_spotrf_batched_ex(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                         cudaStream_t stream, int route);

/*
 * bl_spotrf_route - the route bl_spotrf_batched takes for (n, batch). Host
 * only, needs no GPU. Returns BL_ROUTE_WARP/CTA/BLOCKED, BL_ROUTE_LEFT where
 * the blocked route takes its left-looking order (large batches above n = 256,
 * for 16-byte-aligned batches; judged by the current device's SM count, 152
 * when no device is visible), or 0 when nothing would be launched (n <= 0 or
 * batch <= 0).
 */
int bl_spotrf_route(int n, int batch);

/*
 * bl_spotrf_kernel_info - static resources of the kernel that `route` uses at
 * order n on a 16-byte-aligned batch (route 2 at 64 < n <= 128: the
 * warp-per-tile kernel except at n = 96 and 128, where the shared-memory
 * block kernel runs), as the CUDA runtime reports them (registers per thread, local
 * memory bytes per thread, static shared bytes, dynamic shared bytes the
 * launch asks for, threads per block). Any output pointer may be NULL.
 * Needs a CUDA device. Returns 0, -8 for a route that cannot run n, or a
 * cudaError_t.
 */
int bl_spotrf_kernel_info(int route, int n, int *regs, int *local_bytes, int *static_smem,
                          int *dynamic_smem, int *threads);

/*
 * bl_spotrf_batched_host - bl_spotrf_batched for a batch held in host memory:
 * copy it to the device, factor it there, copy the matrices and info back.
 * The batch is cut into `chunks` slices of whole matrices (chunks <= 0: one
 * per stream); slice c runs on streams[c % nstreams] (its host-to-device
 * copy, its factorization, its device-to-host copies), so with a stream per
 * slice the host-to-device copies run back to back on one copy engine while
 * earlier slices are factored and copied back on the other. Only the batch's
 * own span (matrix b at b*strideA, lda*n floats each, with any gaps between
 * them) is copied; the kernels touch the lower triangles only, so everything
 * else returns unchanged.
 *
 *   A_host, info_host  host memory (page-locked for the copies to overlap),
 *                      same layout as the device call's A and info.
 *   A_dev, info_dev    device work buffers of the same sizes, owned by the
 *                      caller (the library still allocates nothing).
 *   streams, nstreams  the caller's CUDA streams (nstreams >= 1; entries may
 *                      repeat, then their slices serialize). The call does not
 *                      synchronize: the results are on the host once every
 *                      stream is done.
 *
 * For n <= 128 with page-locked host buffers that the device maps (memory
 * from cudaHostAlloc / cudaMallocHost / cudaHostRegister, e.g. a pinned torch
 * tensor) there are no copies: the one kernel of those orders reads each
 * lower-triangle element from host memory and writes its result back there,
 * on streams[0] (A_dev and info_dev are not touched). For larger n on such
 * buffers, kernels copy only the lower triangles: per slice, host -> A_dev,
 * the factorization, then the factors and info back (only A_dev's lower
 * triangles are written; chunks <= 0 here means four slices per stream, and
 * the slices are issued one after another so that copies in and out of
 * different slices overlap). Other buffers take the copy path above.
 *
 * Returns what bl_spotrf_batched returns (argument indices as there, with the
 * device buffers checked as A and info; -11 when streams is NULL or nstreams
 * < 1), or the cudaError_t of a failed copy.
 */
int bl_spotrf_batched_host(float *A_host, int n, int lda, int64_t strideA, int batch,
                           int *info_host, float *A_dev, int *info_dev, int chunks,
                           const cudaStream_t *streams, int nstreams);

/*
 * bl_spotrs_batched - solve A_b X_b = B_b for a strided batch, given the
 * Cholesky factors L_b (A_b = L_b L_b^T, as bl_spotrf_batched leaves them):
 * the forward solve L Y = B, then the backward solve L^T X = Y, each
 * right-hand side column independently (the potrf-then-two-triangular-solves
 * composition of posv on the "BatchLAS perf_blackwell" page; LAPACK SPOTRS
 * with uplo = 'L'). X overwrites B.
 *
 *   L        device pointer to factor 0 (float, column-major); only its lower
 *            triangle (i >= j, i < n) is read; nothing of it is written.
 *   n        order (0 <= n <= BL_SPOTRF_MAX_N).
 *   lda      leading dimension of L, lda >= max(1, n).
 *   strideA  distance in floats between L_b and L_{b+1}; >= lda*n when batch > 1.
 *   B        device pointer to right-hand sides 0 (float, column-major, n x nrhs).
 *            Rows n..ldb-1 of every column and the memory between batches
 *            are never read or written.
 *   nrhs     number of right-hand sides (>= 0).
 *   ldb      leading dimension of B, ldb >= max(1, n).
 *   strideB  distance in floats between B_b and B_{b+1}; >= ldb*nrhs when batch > 1.
 *   batch    number of systems (>= 0).
 *   stream   CUDA stream the work is enqueued on.
 *
 * Ownership and threading as bl_spotrf_batched: no allocation, no sync,
 * stream-ordered, reentrant. Every L_b must be a valid factor (nonzero
 * diagonal); a zero or NaN diagonal gives Inf/NaN solutions, not an error.
 * Returns 0 when enqueued, a negative -i when argument i is invalid (nothing
 * is enqueued; checked in the order -2, -6, -9, -3, -7, -4, -8, -1, -5; -2
 * also when n > BL_SPOTRF_MAX_N), or the cudaError_t of a failed launch.
 * Quick return: nothing is enqueued when batch, n or nrhs is 0.
 */
int bl_spotrs_batched(const float *L, int n, int lda, int64_t strideA, float *B, int nrhs,
                      int ldb, int64_t strideB, int batch, cudaStream_t stream);

/*
 * bl_sposv_batched - factor and solve: A_b = L_b L_b^T in place of A_b (as
 * bl_spotrf_batched, info[b] as there), then for every b with info[b] == 0
 * solve A_b X_b = B_b in place of B_b (as bl_spotrs_batched). Systems whose
 * factorization failed keep B_b unchanged (LAPACK SPOSV returns no solution
 * there). Arguments as the two calls above, info a device pointer to batch
 * ints. Returns 0, a negative argument index (checked in the order -2, -6,
 * -9, -3, -7, -4, -8, -1, -5, -10; -2 also when n > BL_SPOTRF_MAX_N) or a
 * cudaError_t. n == 0 sets info[b] = 0; nrhs == 0 only factors.
 */
int bl_sposv_batched(float *A, int n, int lda, int64_t strideA, float *B, int nrhs, int ldb,
                     int64_t strideB, int batch, int *info, cudaStream_t stream);

/*
 * The uplo = 'U' forms (LAPACK's other storage; also the lower triangle of a
 * row-major matrix, such as a (batch, n, n) row-major tensor). With uplo 'U'
 * or 'u' the factor is A_b = U_b^T U_b, U_b upper triangular with a positive
 * diagonal (U_b = L_b^T of the same symmetric matrix: the same pivots, the
 * same info), and only the upper triangle (i <= j, j < n) of each A_b is read
 * and written; the strict lower triangle, rows n..lda-1 and the gaps stay
 * untouched. The solve reads U_b's upper triangle: U^T Y = B, then U X = Y.
 * uplo 'L' or 'l' is exactly the call without uplo.
 *
 * uplo is argument 1, so every other argument's index is one higher than in
 * the call without it: -1 for an invalid uplo, then the codes of that call
 * minus one, in the same order (bl_spotrf_batched_uplo: -2 A, -3 n, -4 lda,
 * -5 strideA, -6 batch, -7 info, -8 n > BL_SPOTRF_MAX_N; _ex: -9 route or a
 * route that cannot run n, which includes BL_ROUTE_TMEM for 'U';
 * bl_spotrs_batched_uplo: -2 .. -10; bl_sposv_batched_uplo: -2 .. -11).
 * Positive values are cudaError_t codes, as above. Kernels: the same routes
 * and the same arithmetic with transposed addresses (BL_ROUTE_TMEM excepted).
 */
int bl_spotrf_batched_uplo(char uplo, float *A, int n, int lda, int64_t strideA, int batch,
                           int *info, cudaStream_t stream);
int bl_spotrf_batched_uplo_ex(char uplo, float *A, int n, int lda, int64_t strideA, int batch,
                              int *info, cudaStream_t stream, int route);
int bl_spotrs_batched_uplo(char uplo, const float *A, int n, int lda, int64_t strideA, float *B,
                           int nrhs, int ldb, int64_t strideB, int batch, cudaStream_t stream);
int bl_sposv_batched_uplo(char uplo, float *A, int n, int lda, int64_t strideA, float *B,
                          int nrhs, int ldb, int64_t strideB, int batch, int *info,
                          cudaStream_t stream);

/*
 * bl_dpotrf_batched / bl_dpotrf_batched_uplo - the same factorization for a
 * double-precision batch (DPOTRF): A is double*, everything else (layout,
 * lda and strideA in elements, the triangle read and written, info, quick
 * returns, argument indices and their order, stream ordering, ownership) as
 * bl_spotrf_batched and bl_spotrf_batched_uplo. IEEE double arithmetic with
 * FMA contraction, IEEE square root and division. On GB300 the FP64 rate is
 * about 1/70 of the FP32 rate (1.05 against 74.7 TFLOP/s by bl_fma_probe),
 * so these calls are bound by their n^3/3 flops. "BatchLAS perf_blackwell"
 * lists double, complex float and complex double among the element types of
 * its batched potrf (the type columns of its potrf rows); these calls and the
 * two below are those types.
 */
int bl_dpotrf_batched(double *A, int n, int lda, int64_t strideA, int batch, int *info,
                      cudaStream_t stream);
int bl_dpotrf_batched_uplo(char uplo, double *A, int n, int lda, int64_t strideA, int batch,
                           int *info, cudaStream_t stream);

/*
 * bl_cpotrf_batched / bl_cpotrf_batched_uplo - the factorization of a
 * single-precision complex Hermitian batch (CPOTRF): A = L L^H with L lower
 * triangular and a real positive diagonal (uplo 'U': A = U^H U, U = L^H, in
 * the upper triangle). A points at interleaved complex floats (real,
 * imaginary; the layout of std::complex<float> / cuFloatComplex), 8-byte
 * aligned (else -1, or -2 for the uplo form); lda and strideA count complex
 * elements. The imaginary part of the diagonal is not read (taken as zero),
 * and the factor's diagonal is written with a zero imaginary part. Pivots
 * d_j = re(a_jj) - sum_k |l_jk|^2 are tested as in bl_spotrf_batched. All
 * other conventions (info, argument indices, quick returns, ownership,
 * streams) as bl_spotrf_batched / bl_spotrf_batched_uplo.
 */
int bl_cpotrf_batched(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                      cudaStream_t stream);
int bl_cpotrf_batched_uplo(char uplo, float *A, int n, int lda, int64_t strideA, int batch,
                           int *info, cudaStream_t stream);

/*
 * bl_zpotrf_batched / bl_zpotrf_batched_uplo - the same for a
 * double-precision complex batch (ZPOTRF): A points at interleaved complex
 * doubles (std::complex<double> / cuDoubleComplex), 16-byte aligned (else -1,
 * or -2 for the uplo form); everything else as bl_cpotrf_batched.
 */
int bl_zpotrf_batched(double *A, int n, int lda, int64_t strideA, int batch, int *info,
                      cudaStream_t stream);
int bl_zpotrf_batched_uplo(char uplo, double *A, int n, int lda, int64_t strideA, int batch,
                           int *info, cudaStream_t stream);

/*
 * bl_fma_probe - the FMA throughput this device reaches (TFLOP/s, 2 flops an
 * FMA) with eight independent FMA chains a thread, 256 threads a block and
 * eight blocks an SM: the compute peak the factorizations are read against
 * (precision 32 or 64). out: a device pointer to one element of that
 * precision (written only in a case that does not occur; it keeps the chains
 * from being removed). Synchronizes `stream` (it times two launches with
 * events). Returns 0, -1 (precision), -2 (out NULL), -3 (tflops NULL) or a
 * cudaError_t.
 */
int bl_fma_probe(int precision, void *out, double *tflops, cudaStream_t stream);

/*
 * bl_spotrf_workspace_bytes - the workspace bl_spotrf_batched_ws can use for
 * (n, batch): 64 KB (one 128 x 128 float block) per matrix when n > 128, 0
 * otherwise (and for n <= 0, batch <= 0 or n above BL_SPOTRF_MAX_N). Host
 * only.
 *
 * bl_spotrf_batched_ws / bl_spotrf_batched_uplo_ws - bl_spotrf_batched (and
 * its uplo form) with a caller-owned device workspace `work` of `work_bytes`
 * bytes. On the blocked route (n > 128) the panels with at least 256 rows below
 * their 128 x 128 diagonal block are then solved by the inverse of that block
 * (the inverse-based panel solve of "kernelbot-cholesky-930185", changelog
 * section "THE MECHANISM, FOR THE NEXT BUILD": the inverse, computed once per
 * matrix and panel into the workspace, and one tensor-core product per 128 rows
 * instead of a forward substitution); every other step is the same as in
 * bl_spotrf_batched. The workspace holds nothing between calls and may be
 * reused by any later call on the same stream; calls in flight at once on
 * different streams need their own. work = NULL: exactly bl_spotrf_batched.
 * The results agree with bl_spotrf_batched within the same tolerances but not
 * bit for bit (a product by the inverse rounds differently from the
 * substitution), and the explicit inverse makes the panel's accuracy depend on
 * the conditioning of its diagonal block. Returns as bl_spotrf_batched, plus
 * -8 (work not 16-byte aligned) and -9 (work_bytes below
 * bl_spotrf_workspace_bytes(n, batch)); the uplo form moves every negative code
 * down by one (uplo is argument 1).
 */
size_t bl_spotrf_workspace_bytes(int n, int batch);
int bl_spotrf_batched_ws(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                         void *work, size_t work_bytes, cudaStream_t stream);
int bl_spotrf_batched_uplo_ws(char uplo, float *A, int n, int lda, int64_t strideA, int batch,
                              int *info, void *work, size_t work_bytes, cudaStream_t stream);

/* Device memory the library reserves on every GPU that loads it, for
 * bl_spotrf_batched_static (held until the process exits). */
#define BL_SPOTRF_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * bl_spotrf_batched_static - bl_spotrf_batched_ws for callers that cannot
 * allocate device memory where they factor: a library running inside a
 * framework that owns all device memory through an allocator the library
 * cannot reach, a latency-bounded loop that cannot take the device-wide
 * synchronization cudaMalloc and cudaFree may cause, or a process that already
 * holds all the memory it was given. The call allocates nothing: the scratch of
 * the inverse-based panel solve comes from a fixed device array of
 * BL_SPOTRF_STATIC_SCRATCH_BYTES inside the library, so a call whose scratch
 * would exceed it (n > 128 and batch > 256) is rejected with -10 before any
 * work. The caller still owns A and info; arguments, results, info and every
 * other return code are those of bl_spotrf_batched_ws with a workspace.
 *
 * The first call made on a device looks the array's device address up (once
 * per device, on the host, with that device current); make that first call
 * before capturing a stream into a CUDA graph. All calls share the one array,
 * which keeps the last call's contents: every block a call reads it has
 * written first, so nothing needs clearing, but calls that run at the same
 * time on the GPU (on different streams, or from different host threads) race
 * on it and must be ordered by the caller.
 *
 * The pages have no counterpart to this entry point: it exists for the callers
 * above.
 */
int bl_spotrf_batched_static(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                             cudaStream_t stream);

/*
 * bl_debug_fail_first_wait - failure injection, for testing the internal-error
 * path (info[b] = -1) only. While `every` > 0 for a kernel class, every block
 * of that class on the current device whose matrix index b is a multiple of
 * `every` reports its first bounded wait as timed out without waiting and
 * takes the path a real timeout takes: it sets info[b] = -1, lets the copies
 * and tensor-core operations it has already issued finish (bounded), releases
 * its tensor memory and exits; later launches of the same call skip matrix b.
 * Other matrices are factored as usual. every = 0 (the state at load) turns
 * the injection off. Classes: 1 the shared-memory block
 * kernel's bulk-copy load (route 2 at n = 96 and 128 on 16-byte-aligned
 * batches, and the diagonal blocks of route 3), 2 the tensor-core panel solve
 * and 3 the tensor-core trailing update (route 3 on 16-byte-aligned batches),
 * 4 the tensor-memory kernel (route 4), 5 the tensor-core product of the
 * inverse-based panel solve (bl_spotrf_batched_ws), 6 the tensor-core trailing
 * update of the single-precision complex call (bl_cpotrf_batched, n > 128,
 * lower storage, 16-byte-aligned batches), 7 the tensor-core panel solve of
 * the same call. Synchronous with the host; call it
 * while no other work of the library runs. Returns 0, -1 (unknown class), -2
 * (every < 0) or a cudaError_t.
 */
int bl_debug_fail_first_wait(int kernel_class, int every);

/* Version string of the library ("bl_spotrf <major>.<minor> sm_103a"). */
const char *bl_spotrf_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BL_SPOTRF_H */
