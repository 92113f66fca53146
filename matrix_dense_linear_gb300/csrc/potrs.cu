// KS: batched SPOTRS (uplo = 'L'): solve A_b X_b = B_b in place of B_b with
// the Cholesky factor L_b of A_b, as the two triangular solves of the posv
// composition of "BatchLAS perf_blackwell" (potrf, then L Y = B, then
// L^T X = Y; "BatchLAS perf_trsm" fuses the solves for the tiny sizes).
//
// One block of 128 threads per (matrix, group of 32 right-hand sides).
// Rows go in blocks of 32: lane r of every warp owns row r of the current row
// block, warp w owns right-hand sides 8w .. 8w+7, so a thread accumulates 8
// values. Both solves are left-looking over the row blocks:
//   forward   Y_j = L_jj^{-1} (B_j - sum_{i<j} L_ji Y_i)
//   backward  X_j = L_jj^{-T} (Y_j - sum_{i>j} L_ij^T X_i)
// The block products stream a 32 x 32 block of L and the already solved 32 x
// 32 block of Y (or X) through double-buffered shared memory with cp.async
// (L_ji column-major so lane r reads row r; the solution block row-major so a
// warp reads its 8 columns as two 16-byte broadcasts): per k one shared load
// of L, two broadcasts and 8 FMAs. The 32 x 32 triangular solve is one warp
// per 8 columns: lane i scales its row by 1/l_ii and publishes it through a
// warp-private buffer, the lanes below subtract (32 dependent steps, no block
// barrier). Solved blocks are written to B at once and read back (through L2)
// by the later block products of the same thread block.
//
// Rows from n on and right-hand sides from nrhs on are zero (L's diagonal
// there is taken as 1); they are never written. A matrix whose info entry is
// nonzero is left untouched (the posv path).

#include "bl_common.cuh"

namespace bl {
namespace {

constexpr int kT = 128;  // 4 warps x 8 right-hand sides
constexpr int kLd = 36;  // leading dimension of a 32 x 32 block in shared memory

struct TrsShared {
    float L[2][32 * kLd];   // product operand: L block, layout set by the pass
    float S[2][32 * kLd];   // product operand: solved block, [k][c]
    float D[32 * kLd];      // diagonal block, layout set by the pass
    float rcp[32];          // 1 / l_ii of the diagonal block
    float bc[4][2][8];      // per-warp broadcast of one solved row (double-buffered)
};

// 4-byte asynchronous copy that fills zeros when `ok` is false
__device__ __forceinline__ void cp4(float *dst, const float *src, bool ok)
{
    if (ok) cp_async4(dst, src);
    else *dst = 0.0f;
}

// The solved block i (rows 32i.., right-hand sides c0..c0+31) of B into S as
// [k][c]: 8 elements per thread, column-wise coalesced.
__device__ __forceinline__ void stage_solved(float *S, const float *Bb, int ldb, int n, int nrhs,
                                             int i, int c0, int tid)
{
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int idx = tid + kT * e;        // 0 .. 1023
        const int k = idx & 31, c = idx >> 5;  // k fastest: a warp reads one column
        const int row = 32 * i + k, col = c0 + c;
        cp4(S + k * kLd + c, Bb + row + (int64_t)col * ldb, row < n && col < nrhs);
    }
}

// Block (rb, cb) of L (rows 32rb.., columns 32cb..) into Ls.
//   COLMAJOR: Ls[col * kLd + row] (element (row, col) of the block)
//   else:     Ls[row * kLd + col]
template <bool COLMAJOR>
__device__ __forceinline__ void stage_L(float *Ls, const float *Lb, int lda, int n, int rb, int cb,
                                        int tid)
{
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int idx = tid + kT * e;
        const int row = idx & 31, col = idx >> 5;  // row fastest: a warp reads one column
        const int gr = 32 * rb + row, gc = 32 * cb + col;
        float *dst = COLMAJOR ? Ls + col * kLd + row : Ls + row * kLd + col;
        cp4(dst, Lb + gr + (int64_t)gc * lda, gr < n && gc < n && gr >= gc);
    }
}

__global__ void __launch_bounds__(kT, 8)
potrs_kernel(const float *__restrict__ L, int n, int lda, int64_t strideA, float *__restrict__ B,
             int nrhs, int ldb, int64_t strideB, const int *__restrict__ info)
{
    __shared__ __align__(16) TrsShared sm;

    const int64_t mat = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    if (info != nullptr && info[mat] != 0) return;
    const float *Lb = L + mat * strideA;
    float *Bb = B + mat * strideB;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c0 = 32 * (int)blockIdx.y;     // first right-hand side of this block
    const int cw = c0 + 8 * warp;            // this warp's first right-hand side
    const int NB = (n + 31) >> 5;

    float acc[8];

    // ---------------- forward: L Y = B ----------------
#pragma unroll 1
    for (int j = 0; j < NB; ++j) {
        const int row = 32 * j + lane;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            acc[u] = (row < n && cw + u < nrhs) ? Bb[row + (int64_t)(cw + u) * ldb] : 0.0f;
        // block products with the solved blocks i < j (double-buffered)
        if (j > 0) {
            stage_L<true>(sm.L[0], Lb, lda, n, j, 0, tid);
            stage_solved(sm.S[0], Bb, ldb, n, nrhs, 0, c0, tid);
            cp_async_commit();
        }
#pragma unroll 1
        for (int i = 0; i < j; ++i) {
            const int buf = i & 1;
            if (i + 1 < j) {
                stage_L<true>(sm.L[buf ^ 1], Lb, lda, n, j, i + 1, tid);
                stage_solved(sm.S[buf ^ 1], Bb, ldb, n, nrhs, i + 1, c0, tid);
                cp_async_commit();
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const float *Ls = sm.L[buf];
            const float *Ss = sm.S[buf] + 8 * warp;
#pragma unroll 8
            for (int k = 0; k < 32; ++k) {
                const float a = Ls[k * kLd + lane];
                const float4 s0 = *reinterpret_cast<const float4 *>(Ss + k * kLd);
                const float4 s1 = *reinterpret_cast<const float4 *>(Ss + k * kLd + 4);
                acc[0] = fmaf(-a, s0.x, acc[0]); acc[1] = fmaf(-a, s0.y, acc[1]);
                acc[2] = fmaf(-a, s0.z, acc[2]); acc[3] = fmaf(-a, s0.w, acc[3]);
                acc[4] = fmaf(-a, s1.x, acc[4]); acc[5] = fmaf(-a, s1.y, acc[5]);
                acc[6] = fmaf(-a, s1.z, acc[6]); acc[7] = fmaf(-a, s1.w, acc[7]);
            }
            __syncthreads();  // the buffer is restaged two products later
        }
        // the diagonal block, column-major: lane k reads l_(k,i) at D[i*kLd + k]
        stage_L<true>(sm.D, Lb, lda, n, j, j, tid);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        if (tid < 32) {
            const int r = 32 * j + tid;
            sm.rcp[tid] = r < n ? 1.0f / sm.D[tid * kLd + tid] : 1.0f;
        }
        __syncthreads();
        // y_i = acc_i / l_ii on lane i, published; lanes k > i subtract l_ki y_i
#pragma unroll 1
        for (int i = 0; i < 32; ++i) {
            float *bc = sm.bc[warp][i & 1];
            if (lane == i) {
                const float s = sm.rcp[i];
#pragma unroll
                for (int u = 0; u < 8; ++u) acc[u] *= s;
                *reinterpret_cast<float4 *>(bc) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                *reinterpret_cast<float4 *>(bc + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
            }
            __syncwarp();
            if (lane > i) {
                const float4 y0 = *reinterpret_cast<const float4 *>(bc);
                const float4 y1 = *reinterpret_cast<const float4 *>(bc + 4);
                const float l = sm.D[i * kLd + lane];
                acc[0] = fmaf(-l, y0.x, acc[0]); acc[1] = fmaf(-l, y0.y, acc[1]);
                acc[2] = fmaf(-l, y0.z, acc[2]); acc[3] = fmaf(-l, y0.w, acc[3]);
                acc[4] = fmaf(-l, y1.x, acc[4]); acc[5] = fmaf(-l, y1.y, acc[5]);
                acc[6] = fmaf(-l, y1.z, acc[6]); acc[7] = fmaf(-l, y1.w, acc[7]);
            }
        }
        if (row < n) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (cw + u < nrhs) Bb[row + (int64_t)(cw + u) * ldb] = acc[u];
        }
        __syncthreads();  // Y_j is in B before any later product reads it
    }

    // ---------------- backward: L^T X = Y ----------------
#pragma unroll 1
    for (int j = NB - 1; j >= 0; --j) {
        const int row = 32 * j + lane;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            acc[u] = (row < n && cw + u < nrhs) ? Bb[row + (int64_t)(cw + u) * ldb] : 0.0f;
        // block products with the solved blocks i > j: (L_ij)^T X_i, where lane
        // r needs l_(32i+k, 32j+r): L_ij staged row-major (Ls[k*kLd + r])
        if (j + 1 < NB) {
            stage_L<false>(sm.L[0], Lb, lda, n, j + 1, j, tid);
            stage_solved(sm.S[0], Bb, ldb, n, nrhs, j + 1, c0, tid);
            cp_async_commit();
        }
#pragma unroll 1
        for (int i = j + 1; i < NB; ++i) {
            const int buf = (i - j - 1) & 1;
            if (i + 1 < NB) {
                stage_L<false>(sm.L[buf ^ 1], Lb, lda, n, i + 1, j, tid);
                stage_solved(sm.S[buf ^ 1], Bb, ldb, n, nrhs, i + 1, c0, tid);
                cp_async_commit();
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const float *Ls = sm.L[buf];
            const float *Ss = sm.S[buf] + 8 * warp;
#pragma unroll 8
            for (int k = 0; k < 32; ++k) {
                const float a = Ls[k * kLd + lane];
                const float4 s0 = *reinterpret_cast<const float4 *>(Ss + k * kLd);
                const float4 s1 = *reinterpret_cast<const float4 *>(Ss + k * kLd + 4);
                acc[0] = fmaf(-a, s0.x, acc[0]); acc[1] = fmaf(-a, s0.y, acc[1]);
                acc[2] = fmaf(-a, s0.z, acc[2]); acc[3] = fmaf(-a, s0.w, acc[3]);
                acc[4] = fmaf(-a, s1.x, acc[4]); acc[5] = fmaf(-a, s1.y, acc[5]);
                acc[6] = fmaf(-a, s1.z, acc[6]); acc[7] = fmaf(-a, s1.w, acc[7]);
            }
            __syncthreads();
        }
        // the diagonal block, row-major: lane k reads l_(i,k) at D[i*kLd + k]
        stage_L<false>(sm.D, Lb, lda, n, j, j, tid);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        if (tid < 32) {
            const int r = 32 * j + tid;
            sm.rcp[tid] = r < n ? 1.0f / sm.D[tid * kLd + tid] : 1.0f;
        }
        __syncthreads();
        // x_i = acc_i / l_ii on lane i (i from the bottom), lanes k < i subtract l_ik x_i
#pragma unroll 1
        for (int i = 31; i >= 0; --i) {
            float *bc = sm.bc[warp][i & 1];
            if (lane == i) {
                const float s = sm.rcp[i];
#pragma unroll
                for (int u = 0; u < 8; ++u) acc[u] *= s;
                *reinterpret_cast<float4 *>(bc) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                *reinterpret_cast<float4 *>(bc + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
            }
            __syncwarp();
            if (lane < i) {
                const float4 x0 = *reinterpret_cast<const float4 *>(bc);
                const float4 x1 = *reinterpret_cast<const float4 *>(bc + 4);
                const float l = sm.D[i * kLd + lane];
                acc[0] = fmaf(-l, x0.x, acc[0]); acc[1] = fmaf(-l, x0.y, acc[1]);
                acc[2] = fmaf(-l, x0.z, acc[2]); acc[3] = fmaf(-l, x0.w, acc[3]);
                acc[4] = fmaf(-l, x1.x, acc[4]); acc[5] = fmaf(-l, x1.y, acc[5]);
                acc[6] = fmaf(-l, x1.z, acc[6]); acc[7] = fmaf(-l, x1.w, acc[7]);
            }
        }
        if (row < n) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (cw + u < nrhs) Bb[row + (int64_t)(cw + u) * ldb] = acc[u];
        }
        __syncthreads();
    }
}

}  // namespace

int launch_potrs(const float *L, int n, int lda, int64_t strideA, float *B, int nrhs, int ldb,
                 int64_t strideB, int batch, const int *info, cudaStream_t stream)
{
    const dim3 grid((unsigned)batch, (unsigned)((nrhs + 31) / 32));
    return launch_pdl(potrs_kernel, grid, dim3(kT), 0, stream, L, n, lda, strideA, B, nrhs, ldb,
                      strideB, info);
}

int attrs_potrs(cudaFuncAttributes *fa, int *threads, int *dyn_smem)
{
    *threads = kT;
    *dyn_smem = 0;
    return (int)cudaFuncGetAttributes(fa, potrs_kernel);
}

}  // namespace bl
