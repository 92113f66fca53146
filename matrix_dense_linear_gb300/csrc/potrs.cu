// KS: batched SPOTRS: solve A_b X_b = B_b in place of B_b with the Cholesky
// factor L_b of A_b (uplo = 'L'; with uplo = 'U' the factor U_b = L_b^T is
// read from the upper triangle, the same solves), as the two triangular solves of the posv
// composition of "BatchLAS perf_blackwell" (potrf, then L Y = B, then
// L^T X = Y; "BatchLAS perf_trsm" fuses the solves for the tiny sizes).
//
// One block of W warps per (matrix, group of W*C right-hand sides), with
// (W, C) = (1, 1), (1, 2), (1, 4), (1, 8), (2, 8) or (4, 8) picked from nrhs.
// Rows go in blocks of 32: lane r of every warp owns row r of the current row
// block, warp w owns right-hand sides C*w .. C*w+C-1, so a thread accumulates
// C values. Both solves are left-looking over the row blocks:
//   forward   Y_j = L_jj^{-1} (B_j - sum_{i<j} L_ji Y_i)
//   backward  X_j = L_jj^{-T} (Y_j - sum_{i>j} L_ij^T X_i)
// The block products stream a 32 x 32 block of L and the already solved 32 x
// 32 block of Y (or X) through double-buffered shared memory with cp.async
// (L_ji column-major so lane r reads row r; the solution block row-major so a
// warp reads its C columns as broadcasts): per k one shared load of L, the
// broadcasts and C FMAs. The 32 x 32 triangular solve is one warp per C
// columns: lane i scales its row by 1/l_ii and publishes it through a
// warp-private buffer, the lanes below subtract (32 dependent steps, no block
// barrier). Solved blocks are written to B at once and read back (through L2)
// by the later block products of the same thread block.
//
// Rows from n on and right-hand sides from nrhs on are zero (L's diagonal
// there is taken as 1); they are never written. A matrix whose info entry is
// nonzero is left untouched (the posv path).

#include "bl_common.cuh"
#include "launch.cuh"

namespace bl {
namespace {

constexpr int kLd = 36;  // leading dimension of a 32 x 32 block in shared memory

template <int W>
struct TrsShared {
    float L[2][32 * kLd];   // product operand: L block, layout set by the pass
    float S[2][32 * kLd];   // product operand: solved block, [k][c]
    float D[32 * kLd];      // diagonal block, layout set by the pass
    float rcp[32];          // 1 / l_ii of the diagonal block
    float bc[W][2][8];      // per-warp broadcast of one solved row (double-buffered)
};

// 4-byte asynchronous copy that fills zeros when `ok` is false
__device__ __forceinline__ void cp4(float *dst, const float *src, bool ok)
{
    if (ok) cp_async4(dst, src);
    else *dst = 0.0f;
}

// The solved block i (rows 32i.., right-hand sides c0 .. c0+NC-1) of B into S
// as [k][c]; k fastest, so a warp reads one column.
template <int NT, int NC>
__device__ __forceinline__ void stage_solved(float *S, const float *Bb, int ldb, int n, int nrhs,
                                             int i, int c0, int tid)
{
#pragma unroll 4
    for (int e = 0; e < 32 * NC / NT; ++e) {
        const int idx = tid + NT * e;
        const int k = idx & 31, c = idx >> 5;
        const int row = 32 * i + k, col = c0 + c;
        cp4(S + k * kLd + c, Bb + row + (int64_t)col * ldb, row < n && col < nrhs);
    }
}

// Block (rb, cb) of L (rows 32rb.., columns 32cb..) into Ls.
//   COLMAJOR: Ls[col * kLd + row] (element (row, col) of the block)
//   else:     Ls[row * kLd + col]
// A warp reads one column of the block from the lower storage and one row
// from the upper (UP), both contiguous in memory.
template <int NT, bool COLMAJOR, bool UP>
__device__ __forceinline__ void stage_L(float *Ls, const float *Lb, int lda, int n, int rb, int cb,
                                        int tid)
{
#pragma unroll 4
    for (int e = 0; e < 1024 / NT; ++e) {
        const int idx = tid + NT * e;
        const int row = UP ? idx >> 5 : idx & 31, col = UP ? idx & 31 : idx >> 5;
        const int gr = 32 * rb + row, gc = 32 * cb + col;
        float *dst = COLMAJOR ? Ls + col * kLd + row : Ls + row * kLd + col;
        cp4(dst, Lb + lidx<UP>(gr, gc, lda), gr < n && gc < n && gr >= gc);
    }
}

// C consecutive floats of shared memory (16-byte aligned for C >= 4)
template <int C>
__device__ __forceinline__ void lds(const float *p, float (&v)[C])
{
    if constexpr (C == 8) {
        const float4 a = *reinterpret_cast<const float4 *>(p);
        const float4 b = *reinterpret_cast<const float4 *>(p + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else if constexpr (C == 4) {
        const float4 a = *reinterpret_cast<const float4 *>(p);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else if constexpr (C == 2) {
        const float2 a = *reinterpret_cast<const float2 *>(p);
        v[0] = a.x; v[1] = a.y;
    } else {
        v[0] = *p;
    }
}

template <int C>
__device__ __forceinline__ void sts(float *p, const float (&v)[C])
{
    if constexpr (C == 8) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4 *>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
    } else if constexpr (C == 4) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    } else if constexpr (C == 2) {
        *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
    } else {
        *p = v[0];
    }
}

// acc -= a * s over the block product's 32 k (s: C columns of row k)
template <int C>
__device__ __forceinline__ void block_product(float (&acc)[C], const float *Ls, const float *Ss,
                                              int lane)
{
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
        const float a = Ls[k * kLd + lane];
        float sv[C];
        lds<C>(Ss + k * kLd, sv);
#pragma unroll
        for (int u = 0; u < C; ++u) acc[u] = fmaf(-a, sv[u], acc[u]);
    }
}

template <int W, int C, bool UP>
__global__ void __launch_bounds__(32 * W, W == 4 ? 8 : 9)
potrs_kernel(const float *__restrict__ L, int n, int lda, int64_t strideA, float *__restrict__ B,
             int nrhs, int ldb, int64_t strideB, const int *__restrict__ info)
{
    constexpr int NT = 32 * W, NC = W * C;
    __shared__ __align__(16) TrsShared<W> sm;

    const int64_t mat = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    if (info != nullptr && info[mat] != 0) return;
    const float *Lb = L + mat * strideA;
    float *Bb = B + mat * strideB;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c0 = NC * (int)blockIdx.y;     // first right-hand side of this block
    const int cw = c0 + C * warp;            // this warp's first right-hand side
    const int NB = (n + 31) >> 5;

    float acc[C];

    // ---------------- forward: L Y = B ----------------
#pragma unroll 1
    for (int j = 0; j < NB; ++j) {
        const int row = 32 * j + lane;
#pragma unroll
        for (int u = 0; u < C; ++u)
            acc[u] = (row < n && cw + u < nrhs) ? Bb[row + (int64_t)(cw + u) * ldb] : 0.0f;
        // block products with the solved blocks i < j (double-buffered)
        if (j > 0) {
            stage_L<NT, true, UP>(sm.L[0], Lb, lda, n, j, 0, tid);
            stage_solved<NT, NC>(sm.S[0], Bb, ldb, n, nrhs, 0, c0, tid);
            cp_async_commit();
        }
#pragma unroll 1
        for (int i = 0; i < j; ++i) {
            const int buf = i & 1;
            if (i + 1 < j) {
                stage_L<NT, true, UP>(sm.L[buf ^ 1], Lb, lda, n, j, i + 1, tid);
                stage_solved<NT, NC>(sm.S[buf ^ 1], Bb, ldb, n, nrhs, i + 1, c0, tid);
                cp_async_commit();
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            block_product<C>(acc, sm.L[buf], sm.S[buf] + C * warp, lane);
            __syncthreads();  // the buffer is restaged two products later
        }
        // the diagonal block, column-major: lane k reads l_(k,i) at D[i*kLd + k]
        stage_L<NT, true, UP>(sm.D, Lb, lda, n, j, j, tid);
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
                for (int u = 0; u < C; ++u) acc[u] *= s;
                sts<C>(bc, acc);
            }
            __syncwarp();
            if (lane > i) {
                float y[C];
                lds<C>(bc, y);
                const float l = sm.D[i * kLd + lane];
#pragma unroll
                for (int u = 0; u < C; ++u) acc[u] = fmaf(-l, y[u], acc[u]);
            }
        }
        if (row < n) {
#pragma unroll
            for (int u = 0; u < C; ++u)
                if (cw + u < nrhs) Bb[row + (int64_t)(cw + u) * ldb] = acc[u];
        }
        __syncthreads();  // Y_j is in B before any later product reads it
    }

    // ---------------- backward: L^T X = Y ----------------
#pragma unroll 1
    for (int j = NB - 1; j >= 0; --j) {
        const int row = 32 * j + lane;
#pragma unroll
        for (int u = 0; u < C; ++u)
            acc[u] = (row < n && cw + u < nrhs) ? Bb[row + (int64_t)(cw + u) * ldb] : 0.0f;
        // block products with the solved blocks i > j: (L_ij)^T X_i, where lane
        // r needs l_(32i+k, 32j+r): L_ij staged row-major (Ls[k*kLd + r])
        if (j + 1 < NB) {
            stage_L<NT, false, UP>(sm.L[0], Lb, lda, n, j + 1, j, tid);
            stage_solved<NT, NC>(sm.S[0], Bb, ldb, n, nrhs, j + 1, c0, tid);
            cp_async_commit();
        }
#pragma unroll 1
        for (int i = j + 1; i < NB; ++i) {
            const int buf = (i - j - 1) & 1;
            if (i + 1 < NB) {
                stage_L<NT, false, UP>(sm.L[buf ^ 1], Lb, lda, n, i + 1, j, tid);
                stage_solved<NT, NC>(sm.S[buf ^ 1], Bb, ldb, n, nrhs, i + 1, c0, tid);
                cp_async_commit();
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            block_product<C>(acc, sm.L[buf], sm.S[buf] + C * warp, lane);
            __syncthreads();
        }
        // the diagonal block, row-major: lane k reads l_(i,k) at D[i*kLd + k]
        stage_L<NT, false, UP>(sm.D, Lb, lda, n, j, j, tid);
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
                for (int u = 0; u < C; ++u) acc[u] *= s;
                sts<C>(bc, acc);
            }
            __syncwarp();
            if (lane < i) {
                float x[C];
                lds<C>(bc, x);
                const float l = sm.D[i * kLd + lane];
#pragma unroll
                for (int u = 0; u < C; ++u) acc[u] = fmaf(-l, x[u], acc[u]);
            }
        }
        if (row < n) {
#pragma unroll
            for (int u = 0; u < C; ++u)
                if (cw + u < nrhs) Bb[row + (int64_t)(cw + u) * ldb] = acc[u];
        }
        __syncthreads();
    }
}

template <int W, int C>
int launch_wc(const float *L, int n, int lda, int64_t strideA, float *B, int nrhs, int ldb,
              int64_t strideB, int batch, const int *info, cudaStream_t stream, bool upper)
{
    const dim3 grid((unsigned)batch, (unsigned)((nrhs + W * C - 1) / (W * C)));
    if (upper)
        return launch_pdl(potrs_kernel<W, C, true>, grid, dim3(32 * W), 0, stream, L, n, lda,
                          strideA, B, nrhs, ldb, strideB, info);
    return launch_pdl(potrs_kernel<W, C, false>, grid, dim3(32 * W), 0, stream, L, n, lda,
                      strideA, B, nrhs, ldb, strideB, info);
}

}  // namespace

// Right-hand sides per block from nrhs: the narrowest shape that holds them,
// up to 32 (4 warps x 8) per block.
int launch_potrs(const float *L, int n, int lda, int64_t strideA, float *B, int nrhs, int ldb,
                 int64_t strideB, int batch, const int *info, cudaStream_t stream, bool upper)
{
#define BL_POTRS_ARGS L, n, lda, strideA, B, nrhs, ldb, strideB, batch, info, stream, upper
    if (nrhs <= 1) return launch_wc<1, 1>(BL_POTRS_ARGS);
    if (nrhs <= 2) return launch_wc<1, 2>(BL_POTRS_ARGS);
    if (nrhs <= 4) return launch_wc<1, 4>(BL_POTRS_ARGS);
    if (nrhs <= 8) return launch_wc<1, 8>(BL_POTRS_ARGS);
    if (nrhs <= 16) return launch_wc<2, 8>(BL_POTRS_ARGS);
    return launch_wc<4, 8>(BL_POTRS_ARGS);
#undef BL_POTRS_ARGS
}

int attrs_potrs(cudaFuncAttributes *fa, int *threads, int *dyn_smem)
{
    *threads = 128;
    *dyn_smem = 0;
    return (int)cudaFuncGetAttributes(fa, potrs_kernel<4, 8, false>);
}

}  // namespace bl
