// Host-side launchers of the kernels of libbl_spotrf and the info convention
// of a launch (internal, not installed).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace bl {

// One-time setup per device (a kernel's function attributes belong to the
// context of the device they were set on): run(f) calls f once for the
// current device and returns its result there on every call.
class DeviceOnce {
public:
    template <typename F>
    int run(F &&f)
    {
        int dev = 0;
        const cudaError_t g = cudaGetDevice(&dev);
        if (g != cudaSuccess) return (int)g;
        if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
        std::call_once(flag_[dev], [&] { err_[dev] = f(); });
        return (int)err_[dev];
    }

private:
    static constexpr int kMaxDevices = 64;
    std::once_flag flag_[kMaxDevices];
    cudaError_t err_[kMaxDevices] = {};
};

// info handling of one launch over a strided batch.
//   info_off < 0 : the launch factors whole matrices and writes info[b]
//                  unconditionally (0 or the failing pivot).
//   info_off >= 0: the launch factors the diagonal block at (info_off,
//                  info_off) of a larger matrix; it skips matrices whose
//                  info[b] is already nonzero and writes info[b] only on a
//                  failure, as info_off + local index.
struct InfoMode {
    int off;
};

// `upper`: the factor is stored in the upper triangle (uplo = 'U', see lidx).
int launch_warp(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                cudaStream_t stream, bool upper);
// no_bulk: A may be host memory the device maps (no bulk copies then)
int launch_cta(float *A, int n, int lda, int64_t strideA, int batch, int *info,
               cudaStream_t stream, InfoMode mode, bool upper, bool no_bulk = false);
int launch_tmem(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                cudaStream_t stream, InfoMode mode);
// W: the caller's workspace for the inverse-based panel solve (kInvBytes per
// matrix, 16-byte aligned), or nullptr (substitution only)
// whether the automatic blocked route takes the left-looking order (aligned
// panels, no workspace), and the SM count it judges by (152 when no device is
// visible)
bool left_pays(int n, int batch, int sms);
int sm_count_or_default();
// the left-looking schedule of the same kernels (BL_ROUTE_LEFT)
int launch_left(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                cudaStream_t stream, bool upper);
int launch_blocked(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                   cudaStream_t stream, bool upper, float *W = nullptr);
constexpr size_t kInvBytes = 128 * 128 * sizeof(float);
// the argument checks of bl_spotrf_batched (0 or a negative argument index)
int check_potrf_args(const void *A, int n, int lda, int64_t strideA, int batch, const int *info);
// The panel solve by the inverse of the diagonal block (trsm_inv.cu): W[b] =
// L11^{-1} of matrix b, then L21 = A21 W^T on the tensor cores. Returns 1 when
// A or W is not 16-byte aligned (the caller's substitution path).
int launch_trsm_inv(float *A, int n, int lda, int64_t strideA, int batch, int *info, int c0,
                    float *W, cudaStream_t stream, bool upper);

// A22 -= L21 L21^T with k columns c0 .. c0+nk-1 (nk = 128: one panel, 256: two
// panels at once) over the trailing matrix from c0 + nk: every lower tile, or
// with `narrow` only its first tile column. Returns 1 when the panels are not
// 16-byte aligned (the caller's FP32 path), -1 on a bad nk.
int launch_syrk_tc(float *A, int n, int lda, int64_t strideA, int batch, int *info, int c0,
                   int nk, bool narrow, cudaStream_t stream, bool upper);
int attrs_syrk_tc(cudaFuncAttributes *fa);
// fused: also A22 -= L21 L21^T (only when the trailing matrix is one tile, m <= 128)
int launch_trsm_tc(float *A, int n, int lda, int64_t strideA, int batch, int *info, int c0,
                   cudaStream_t stream, bool upper, bool fused);

// Failure injection for the test of the give-up path. Each kernel file with
// bounded waits keeps its own device flag (every file is a device module of
// its own) on the current device; while it is positive, every block of that
// file's kernels whose matrix index is a multiple of it reports its first
// bounded wait as timed out without waiting, and so takes the path a real
// timeout takes: info = -1, the copies and MMAs it has in flight drained
// (bounded), tensor memory released. Zero in normal runs.
int set_fail_first_wait_cta(int every);      // K2's bulk-copy load
int set_fail_first_wait_trsm_tc(int every);  // tensor-core panel solve
int set_fail_first_wait_syrk_tc(int every);  // tensor-core trailing update
int set_fail_first_wait_tmem(int every);     // K2t
int set_fail_first_wait_trsm_inv(int every); // the inverse-based panel solve's GEMM
int set_fail_first_wait_cherk_tc(int every); // the complex tensor-core trailing update
int set_fail_first_wait_ctrsm_tc(int every); // the complex tensor-core panel solve

int launch_dpotrf(double *A, int n, int lda, int64_t strideA, int batch, int *info,
                  cudaStream_t stream, bool upper);
// A: interleaved complex float (re, im); lda and strideA in complex elements
// CPOTRF for n <= 64 in registers: a lane per row (n <= 32: 1, 2 or 4 matrices a warp;
// above: two warps a matrix)
int launch_cpotrf_warp(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                       cudaStream_t stream, bool upper);
// CPOTRF for 64 < n <= 128: a warp per 32 x 32 tile of the lower triangle
int launch_cpotrf_tiles(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                        cudaStream_t stream, bool upper, int info_off = -1);
// the same schedule on real input (64 < n <= 128), a measured alternative to K2
int launch_spotrf_tiles(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                        cudaStream_t stream, bool upper, int info_off = -1);
int attrs_tiles(int n, cudaFuncAttributes *fa, int *threads, int *dyn_smem);
// A22 -= L21 L21^H of the complex blocked path (interleaved complex floats,
// lda and strideA in complex elements; upper: the same on U = L^H) on the
// tensor cores; returns 1 when the panels are not 16-byte aligned (the
// caller's FP32 path)
int launch_cherk_tc(float *A, int n, int lda, int64_t strideA, int batch, int *info, int c0,
                    cudaStream_t stream, bool upper);
// lower triangles of nb matrices (and, when info_src is given, their info
// entries) from src to dst, both in the same strided layout; either side may
// be mapped host memory
int launch_tri_copy(const float *src, float *dst, int n, int lda, int64_t strideA, int nb,
                    const int *info_src, int *info_dst, cudaStream_t stream);
// L21 = A21 L11^{-H} of the complex blocked path (the same conventions) with
// the block updates on the tensor cores; returns 1 when the panels are not
// 16-byte aligned (the caller's FP32 kernel)
int launch_ctrsm_tc(float *A, int n, int lda, int64_t strideA, int batch, int *info, int c0,
                    cudaStream_t stream, bool upper);
int launch_cpotrf(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                  cudaStream_t stream, bool upper);
// A: interleaved complex double; lda and strideA in complex elements
int launch_zpotrf(double *A, int n, int lda, int64_t strideA, int batch, int *info,
                  cudaStream_t stream, bool upper);
int launch_potrs(const float *L, int n, int lda, int64_t strideA, float *B, int nrhs, int ldb,
                 int64_t strideB, int batch, const int *info, cudaStream_t stream, bool upper);
int attrs_potrs(cudaFuncAttributes *fa, int *threads, int *dyn_smem);
int attrs_warp(int n, cudaFuncAttributes *fa, int *threads, int *dyn_smem);
int attrs_cta(int n, cudaFuncAttributes *fa, int *threads, int *dyn_smem);
int attrs_tmem(int n, cudaFuncAttributes *fa, int *threads, int *dyn_smem);
int attrs_blocked(int n, cudaFuncAttributes *fa, int *threads, int *dyn_smem);

}  // namespace bl
