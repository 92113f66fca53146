// Device helpers shared by the kernels of libbl_spotrf (not installed); the
// host-side launcher declarations are in launch.cuh.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bl {

// Pivot test of batched SPOTRF: a pivot passes only when it is > 0, so zero,
// negative and NaN pivots all fail (the first failure's 1-based index is info).
// A positive pivot below FLT_MIN (a subnormal) fails too: the reciprocal root
// below flushes it to zero, so it is a zero pivot in single precision, and a
// matrix that reports info = 0 never carries the infinite root it would give.
// One IEEE comparison: d >= FLT_MIN is false for subnormals, zero, negatives
// and NaN, true for normal positive numbers and +Inf.
__device__ __forceinline__ bool pivot_ok(float d) { return d >= 1.17549435e-38f; }

// Whether the block's matrix has already failed (info[mat] != 0), read once
// by thread 0 and shared through the block, so that every thread takes the
// same branch even while a sibling block of the same matrix writes info[mat]
// (a tile or row block that gave up sets it to -1). Every thread of the block
// must call it (it contains a block barrier).
__device__ __forceinline__ bool block_skip(const int *info, int64_t mat)
{
    __shared__ int flag;
    if (threadIdx.x == 0) flag = *(volatile const int *)(info + mat);
    __syncthreads();
    return flag != 0;
}

// Failure injection for the test of the give-up path: a kernel file with
// bounded waits keeps a device flag `every` (0 in normal runs); when it is
// positive, the blocks of matrices whose index is a multiple of it report their
// first bounded wait as timed out.
__device__ __forceinline__ bool injected_failure(int every, int64_t mat)
{
    return every > 0 && mat % every == 0;
}

// 1/sqrt(d) with the hardware approximation (about 2 ulp), the one operation on
// the per-column chain; the pages' measurements put IEEE sqrt + divide there
// at ~25 instructions ("kernelbot-cholesky-930185", chol_diag kernel comment).
// The flush-to-zero form is one instruction on the chain (measured: the
// 128 x 128 block factor 8 % faster); a positive pivot below FLT_MIN counts as
// 0 here (rsqrt = +Inf), which pivot_ok matches by failing that pivot.
__device__ __forceinline__ float rsqrt_approx(float d) {
    float r;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

// sqrt(d) with the hardware approximation; sqrt(+Inf) = +Inf, which keeps an
// infinite pivot's column at l_ij = a_ij * rsqrt(Inf) = 0 like the definition.
__device__ __forceinline__ float sqrt_approx(float d) {
    float r;
    asm("sqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

// Asynchronous global -> shared copies (cp.async): every copy of a thread can
// be in flight at once, with no register holding the value.
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
// Same copies with a byte count: bytes past src_bytes are filled with zeros
// (src_bytes = 0 reads nothing and zero-fills the destination).
__device__ __forceinline__ void cp_async4_zfill(void *smem, const void *gmem, int src_bytes) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(s), "l"(gmem),
                 "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async16_zfill(void *smem, const void *gmem, int src_bytes) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem),
                 "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Where the factor lives. uplo = 'L': A = L L^T, l_ik (i >= k) at A[i + k lda],
// the column-major lower triangle. uplo = 'U': A = U^T U with U = L^T, so the
// same number l_ik = u_ki sits at A[k + i lda], the column-major upper
// triangle (equivalently the lower triangle of the row-major matrix). Every
// kernel computes L and only its addressing depends on the storage.
template <bool UP>
__device__ __forceinline__ int64_t lidx(int i, int k, int lda)
{
    return UP ? (int64_t)k + (int64_t)i * lda : (int64_t)i + (int64_t)k * lda;
}

// Programmatic dependent launch. Kernels launched with launch_pdl may start
// while the previous kernel in the stream is still running; they call
// pdl_wait() before their first access to global memory (it returns once the
// previous grid has completed and its writes are visible) and pdl_trigger()
// to let the next kernel start launching early.
// Named barrier 1..15 over nthreads threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace bl
