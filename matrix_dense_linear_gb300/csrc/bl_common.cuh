// Internal declarations shared by the kernels of libbl_spotrf (not installed).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bl {

// Pivot test of batched SPOTRF: a pivot passes only when it is > 0, so zero,
// negative and NaN pivots all fail (the first failure's 1-based index is info).
__device__ __forceinline__ bool pivot_ok(float d) { return d > 0.0f; }

// 1/sqrt(d) with the hardware approximation (about 2 ulp), the one operation on
// the per-column chain; the pages' measurements put IEEE sqrt + divide there
// at ~25 instructions ("kernelbot-cholesky-930185", chol_diag kernel comment).
__device__ __forceinline__ float rsqrt_approx(float d) {
    float r;
    asm("rsqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

// sqrt(d) with the hardware approximation; sqrt(+Inf) = +Inf, which keeps an
// infinite pivot's column at l_ij = a_ij * rsqrt(Inf) = 0 like the definition.
__device__ __forceinline__ float sqrt_approx(float d) {
    float r;
    asm("sqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

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

int launch_warp(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                cudaStream_t stream);
int launch_cta(float *A, int n, int lda, int64_t strideA, int batch, int *info,
               cudaStream_t stream, InfoMode mode);
int launch_blocked(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                   cudaStream_t stream);

int attrs_warp(int n, cudaFuncAttributes *fa, int *threads, int *dyn_smem);
int attrs_cta(int n, cudaFuncAttributes *fa, int *threads, int *dyn_smem);
int attrs_blocked(int n, cudaFuncAttributes *fa, int *threads, int *dyn_smem);

}  // namespace bl
