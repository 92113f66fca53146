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
constexpr int kWaveMaxN = 1024;  // the wavefront form: a warp per row block, 32 warps at most
constexpr int kRegMaxN = 64;     // the register form, several right-hand sides

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

// ---------------------------------------------------------------------------
// Wavefront form (one right-hand side, n <= 1024): one block of NB =
// ceil(n / 32) warps per system, warp i owning row block i (lane = row). Both
// solves run as a wavefront over the diagonal blocks with one block barrier a
// step:
//   forward step s:  warp s solves Y_s = L_ss^{-1} b_s and publishes it;
//                    every warp i > s subtracts L_is Y_s from its b_i
//   backward step s: warp s solves X_s = L_ss^{-T} y_s, publishes and stores
//                    it; every warp i < s subtracts L_si^T X_s
// so the block products of a step run on all warps at once and a system's
// critical path is the chain of 2 NB diagonal solves, not the ~n^2 / 512 block
// products of the left-looking form above. Inside a diagonal solve each solved
// entry goes to the other lanes by a warp shuffle (one right-hand side: one
// value a step). The L block a warp needs at the next step is loaded into
// registers while the current step's solve runs; the warp's own diagonal block
// stays in shared memory (row r at D[33 r]); Y never leaves the chip (the
// backward pass starts from the warp's own y_i). Measured against the
// left-looking form with several right-hand sides a block, the wavefront
// loses (most of a system's warps wait at the barriers while one solves, and
// fewer systems fit an SM), so it takes one right-hand side only.

// lc[k] = element (r0 + lane, c0 + k) of L when ROWS (lane = row of L), else
// element (r0 + k, c0 + lane); zero outside the matrix. The memory layout of
// the storage decides which of the two is contiguous per lane (VEC: 16-byte
// loads there when the whole block is inside).
template <bool UP, bool VEC, bool ROWS>
__device__ __forceinline__ void load_block(float (&lc)[32], const float *Lb, int lda, int n, int r0,
                                           int c0, int lane)
{
    // per lane: the fixed index and the 32 running ones
    const int fixed = (ROWS ? r0 : c0) + lane;
    const int run0 = ROWS ? c0 : r0;
    const bool fv = fixed < n;
    // contiguous per lane: lower storage with the running index a row (the
    // lane a column), upper storage with the running index a column
    constexpr bool contig = UP ? ROWS : !ROWS;
    if constexpr (contig) {
        // element (run0 + k, fixed) [lower] or (fixed, run0 + k) [upper] at
        // run0 + k + fixed * lda
        const float *p = Lb + run0 + (int64_t)(fv ? fixed : 0) * lda;
        if (VEC && fv && run0 + 32 <= n) {
#pragma unroll
            for (int k = 0; k < 32; k += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(p + k);
                lc[k] = v.x; lc[k + 1] = v.y; lc[k + 2] = v.z; lc[k + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) lc[k] = fv && run0 + k < n ? p[k] : 0.0f;
        }
    } else {
        // element (fixed, run0 + k) [lower] or (run0 + k, fixed) [upper] at
        // fixed + (run0 + k) * lda: coalesced over the lanes
        const float *p = Lb + (fv ? fixed : 0) + (int64_t)run0 * lda;
#pragma unroll
        for (int k = 0; k < 32; ++k) lc[k] = fv && run0 + k < n ? p[(int64_t)k * lda] : 0.0f;
    }
}

template <int MAXW, bool UP, bool VEC>
__global__ void __launch_bounds__(32 * MAXW, 32 / MAXW)
potrs_wave_kernel(const float *__restrict__ L, int n, int lda, int64_t strideA, float *__restrict__ B,
                  int64_t strideB, const int *__restrict__ info)
{
    extern __shared__ __align__(16) float wsm[];
    const int NB = (n + 31) >> 5;
    const int64_t sys = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    if (info != nullptr && info[sys] != 0) return;
    const float *Lb = L + sys * strideA;
    float *Bb = B + sys * strideB;
    const int tid = threadIdx.x, i = tid >> 5, lane = tid & 31;
    const int row = 32 * i + lane;
    const bool rv = row < n;
    float *D = wsm + i * (32 * 33);  // D[33 r + k] = L(32i + r, 32i + k), k <= r (else 0)
    float *Ys = wsm + NB * (32 * 33);  // [2][32]: the block published last

    // the warp's diagonal block (rows past n: the identity) and its entries of b
#pragma unroll 4
    for (int k = 0; k < 32; ++k) {
        const int col = 32 * i + k;
        D[lane * 33 + k] = rv && k <= lane ? Lb[lidx<UP>(row, col, lda)]
                                           : (k == lane ? 1.0f : 0.0f);
    }
    float acc = rv ? Bb[row] : 0.0f;
    float lc[32];
    if (i > 0) load_block<UP, VEC, true>(lc, Lb, lda, n, 32 * i, 0, lane);
    __syncwarp();
    const float rinv = 1.0f / D[lane * 33 + lane];

    // ---------------- forward: L y = b ----------------
#pragma unroll 1
    for (int s = 0; s < NB; ++s) {
        float *Y = Ys + (s & 1) * 32;
        if (i == s) {
            // y_k = acc_k / l_kk from lane k; lanes r > k subtract l_rk y_k
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float l = D[lane * 33 + k];
                const float yk = __shfl_sync(0xffffffffu, acc * rinv, k);
                acc = lane == k ? yk : (lane > k ? fmaf(-l, yk, acc) : acc);
            }
            Y[lane] = acc;
        }
        __syncthreads();
        if (i > s) {
#pragma unroll
            for (int k = 0; k < 32; ++k) acc = fmaf(-lc[k], Y[k], acc);
            if (i > s + 1) load_block<UP, VEC, true>(lc, Lb, lda, n, 32 * i, 32 * (s + 1), lane);
        }
    }

    // ---------------- backward: L^T x = y (acc holds y_i) ----------------
    if (i < NB - 1) load_block<UP, VEC, false>(lc, Lb, lda, n, 32 * (NB - 1), 32 * i, lane);
#pragma unroll 1
    for (int s = NB - 1; s >= 0; --s) {
        float *X = Ys + (s & 1) * 32;
        if (i == s) {
            // x_k = acc_k / l_kk from lane k (k from the bottom); lanes r < k subtract l_kr x_k
#pragma unroll
            for (int k = 31; k >= 0; --k) {
                const float l = D[k * 33 + lane];
                const float xk = __shfl_sync(0xffffffffu, acc * rinv, k);
                acc = lane == k ? xk : (lane < k ? fmaf(-l, xk, acc) : acc);
            }
            X[lane] = acc;
            if (rv) Bb[row] = acc;
        }
        __syncthreads();
        if (i < s) {
#pragma unroll
            for (int k = 0; k < 32; ++k) acc = fmaf(-lc[k], X[k], acc);
            if (i < s - 1) load_block<UP, VEC, false>(lc, Lb, lda, n, 32 * (s - 1), 32 * i, lane);
        }
    }
}

size_t wave_smem(int n)
{
    const int NB = (n + 31) / 32;
    return (size_t)NB * 32 * 33 * 4 + (size_t)2 * 32 * 4;
}

template <int MAXW, bool UP, bool VEC>
int launch_wave_t(const float *L, int n, int lda, int64_t strideA, float *B, int64_t strideB,
                  int batch, const int *info, cudaStream_t stream)
{
    static DeviceOnce attrs;
    if (const int e = attrs.run([] {
            return cudaFuncSetAttribute(potrs_wave_kernel<MAXW, UP, VEC>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)wave_smem(32 * MAXW));
        }))
        return e;
    const int NB = (n + 31) / 32;
    return launch_pdl(potrs_wave_kernel<MAXW, UP, VEC>, dim3((unsigned)batch), dim3(32 * NB),
                      wave_smem(n), stream, L, n, lda, strideA, B, strideB, info);
}

template <int MAXW>
int launch_wave(const float *L, int n, int lda, int64_t strideA, float *B, int64_t strideB,
                int batch, const int *info, cudaStream_t stream, bool upper)
{
    const bool vec = ((reinterpret_cast<uintptr_t>(L) & 15) == 0) && (lda & 3) == 0 &&
                     (strideA & 3) == 0;
#define BL_WAVE_ARGS L, n, lda, strideA, B, strideB, batch, info, stream
    if (upper)
        return vec ? launch_wave_t<MAXW, true, true>(BL_WAVE_ARGS)
                   : launch_wave_t<MAXW, true, false>(BL_WAVE_ARGS);
    return vec ? launch_wave_t<MAXW, false, true>(BL_WAVE_ARGS)
               : launch_wave_t<MAXW, false, false>(BL_WAVE_ARGS);
#undef BL_WAVE_ARGS
}

// ---------------------------------------------------------------------------
// Register form (several right-hand sides, n <= 1024): one warp per (system,
// C right-hand sides), lane = row of the current 32-row block, the two solves
// left-looking over the row blocks like the form above, but with the L blocks
// taken straight into registers (lane r holds row r of L_ji for the forward
// products, column r of L_ij for the backward ones: the loads of the
// wavefront form, coalesced or 16 bytes a lane), the next one fetched while
// the current one is applied, and the solved blocks kept in shared memory as
// [row][right-hand side] and read as 16-byte broadcasts. No block barrier and
// no staging copies: a block product is 32 register values times C broadcast
// columns. The diagonal blocks are solved by substitution with each solved
// row broadcast by warp shuffles. It takes n <= 64, where the shared-memory
// form's staging and barriers cost more than its two blocks of products.

// acc -= lc (32 entries of this lane's row) times the solved rows S[k][0..C)
template <int C>
__device__ __forceinline__ void reg_product(float (&acc)[C], const float (&lc)[32], const float *S)
{
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        float s[C];
        lds<C>(S + k * C, s);
#pragma unroll
        for (int u = 0; u < C; ++u) acc[u] = fmaf(-lc[k], s[u], acc[u]);
    }
}

template <int C, bool UP, bool VEC>
__global__ void __launch_bounds__(32)
potrs_reg_kernel(const float *__restrict__ L, int n, int lda, int64_t strideA, float *__restrict__ B,
                 int nrhs, int ldb, int64_t strideB, int G, const int *__restrict__ info)
{
    extern __shared__ __align__(16) float Ssm[];  // [n rounded to 32][C]
    const int NB = (n + 31) >> 5;
    const int64_t sys = blockIdx.x / G;
    const int c0 = C * (int)(blockIdx.x % G);
    pdl_wait();
    pdl_trigger();
    if (info != nullptr && info[sys] != 0) return;
    const float *Lb = L + sys * strideA;
    float *Bb = B + sys * strideB;
    const int lane = threadIdx.x;
    const unsigned full = 0xffffffffu;

    float acc[C], lc[32], ln[32];
    // ---------------- forward: L Y = B ----------------
#pragma unroll 1
    for (int j = 0; j < NB; ++j) {
        const int row = 32 * j + lane;
        const bool rv = row < n;
#pragma unroll
        for (int u = 0; u < C; ++u)
            acc[u] = rv && c0 + u < nrhs ? Bb[row + (int64_t)(c0 + u) * ldb] : 0.0f;
        if (j > 0) load_block<UP, VEC, true>(lc, Lb, lda, n, 32 * j, 0, lane);
#pragma unroll 1
        for (int i = 0; i < j; ++i) {
            // L_j,i+1 (or the diagonal block's row after the last product)
            load_block<UP, VEC, true>(ln, Lb, lda, n, 32 * j, 32 * (i + 1), lane);
            reg_product<C>(acc, lc, Ssm + 32 * i * C);
#pragma unroll
            for (int k = 0; k < 32; ++k) lc[k] = ln[k];
        }
        if (j == 0) load_block<UP, VEC, true>(lc, Lb, lda, n, 0, 0, lane);
        // lc: row `lane` of L_jj; y_k = acc_k / l_kk from lane k, lanes r > k
        // subtract l_rk y_k
        const float rinv = rv ? 1.0f / Lb[lidx<UP>(row, row, lda)] : 1.0f;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
#pragma unroll
            for (int u = 0; u < C; ++u) {
                const float yk = __shfl_sync(full, acc[u] * rinv, k);
                acc[u] = lane == k ? yk : (lane > k ? fmaf(-lc[k], yk, acc[u]) : acc[u]);
            }
        }
        sts<C>(Ssm + row * C, acc);
        __syncwarp();
    }

    // ---------------- backward: L^T X = Y ----------------
#pragma unroll 1
    for (int j = NB - 1; j >= 0; --j) {
        const int row = 32 * j + lane;
        const bool rv = row < n;
        lds<C>(Ssm + row * C, acc);
        if (j + 1 < NB) load_block<UP, VEC, false>(lc, Lb, lda, n, 32 * (j + 1), 32 * j, lane);
#pragma unroll 1
        for (int i = j + 1; i < NB; ++i) {
            // L_i+1,j, or column `lane` of L_jj after the last product
            load_block<UP, VEC, false>(ln, Lb, lda, n, i + 1 < NB ? 32 * (i + 1) : 32 * j, 32 * j,
                                       lane);
            reg_product<C>(acc, lc, Ssm + 32 * i * C);
#pragma unroll
            for (int k = 0; k < 32; ++k) lc[k] = ln[k];
        }
        if (j + 1 == NB) load_block<UP, VEC, false>(lc, Lb, lda, n, 32 * j, 32 * j, lane);
        // lc: column `lane` of L_jj; x_k = acc_k / l_kk from lane k (from the
        // bottom), lanes r < k subtract l_kr x_k
        const float rinv = rv ? 1.0f / Lb[lidx<UP>(row, row, lda)] : 1.0f;
#pragma unroll
        for (int k = 31; k >= 0; --k) {
#pragma unroll
            for (int u = 0; u < C; ++u) {
                const float xk = __shfl_sync(full, acc[u] * rinv, k);
                acc[u] = lane == k ? xk : (lane < k ? fmaf(-lc[k], xk, acc[u]) : acc[u]);
            }
        }
        __syncwarp();  // every lane has read block j's Y before it is overwritten
        sts<C>(Ssm + row * C, acc);
        if (rv) {
#pragma unroll
            for (int u = 0; u < C; ++u)
                if (c0 + u < nrhs) Bb[row + (int64_t)(c0 + u) * ldb] = acc[u];
        }
        __syncwarp();
    }
}

template <int C, bool UP, bool VEC>
int launch_reg_t(const float *L, int n, int lda, int64_t strideA, float *B, int nrhs, int ldb,
                 int64_t strideB, int batch, const int *info, cudaStream_t stream)
{
    const size_t smem = (size_t)((n + 31) / 32) * 32 * C * 4;
    static DeviceOnce attrs;
    if (const int e = attrs.run([] {
            return cudaFuncSetAttribute(potrs_reg_kernel<C, UP, VEC>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kRegMaxN * C * 4);
        }))
        return e;
    const int G = (nrhs + C - 1) / C;
    const int64_t blocks = (int64_t)batch * G;
    if (blocks > 0x7fffffffLL) return (int)cudaErrorInvalidConfiguration;
    return launch_pdl(potrs_reg_kernel<C, UP, VEC>, dim3((unsigned)blocks), dim3(32), smem, stream,
                      L, n, lda, strideA, B, nrhs, ldb, strideB, G, info);
}

template <int C>
int launch_reg(const float *L, int n, int lda, int64_t strideA, float *B, int nrhs, int ldb,
               int64_t strideB, int batch, const int *info, cudaStream_t stream, bool upper)
{
    const bool vec = ((reinterpret_cast<uintptr_t>(L) & 15) == 0) && (lda & 3) == 0 &&
                     (strideA & 3) == 0;
#define BL_REG_ARGS L, n, lda, strideA, B, nrhs, ldb, strideB, batch, info, stream
    if (upper)
        return vec ? launch_reg_t<C, true, true>(BL_REG_ARGS)
                   : launch_reg_t<C, true, false>(BL_REG_ARGS);
    return vec ? launch_reg_t<C, false, true>(BL_REG_ARGS)
               : launch_reg_t<C, false, false>(BL_REG_ARGS);
#undef BL_REG_ARGS
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
    // one right-hand side: the wavefront form (8, 16 or 32 warps at most, for
    // 64 registers a thread); the left-looking form otherwise
    if (nrhs == 1 && n <= kWaveMaxN) {
        const int NB = (n + 31) / 32;
        if (NB <= 8) return launch_wave<8>(L, n, lda, strideA, B, strideB, batch, info, stream, upper);
        if (NB <= 16)
            return launch_wave<16>(L, n, lda, strideA, B, strideB, batch, info, stream, upper);
        return launch_wave<32>(L, n, lda, strideA, B, strideB, batch, info, stream, upper);
    }
    // several right-hand sides: the register form up to n = 64, the
    // left-looking shared-memory form above (measured on GB300: n = 64 x 1024
    // with 8 right-hand sides 16.1 against 28.5 us, 32 with 32 19.3 against
    // 21.0 us; from n = 128 on the register form loses, 256 x 4096 with 16
    // 927 against 788 us: a warp's chain of block products waits on its L
    // loads, and each group of eight right-hand sides reads L again)
    if (n <= kRegMaxN) {
        if (nrhs <= 2) return launch_reg<2>(BL_POTRS_ARGS);
        if (nrhs <= 4) return launch_reg<4>(BL_POTRS_ARGS);
        return launch_reg<8>(BL_POTRS_ARGS);
    }
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
