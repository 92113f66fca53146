// DPOTRF: batched double-precision Cholesky, the same operation as the
// single-precision path (A = L L^T, or A = U^T U in the upper triangle; info
// = first pivot with !(d > 0)) for a double batch. "BatchLAS perf_blackwell"
// lists double among the types of its batched potrf (the type columns of its
// potrf rows).
//
// On this GPU the FP64 pipe runs at about 1/66 of the FP32 rate (an FMA
// probe: 1.06 against 70 TFLOP/s), so a double factorization is bound by its
// FMA count and nothing else: one warp issuing independent FP64 FMAs keeps an
// SM's FP64 pipe busy. The kernels here are therefore the plain forms, each
// doing only the FMAs of the lower triangle, with IEEE sqrt and division:
//   dpotrf_cta_kernel   n <= 128 (and the 128 x 128 diagonal blocks of larger
//                       n): the block's lower triangle in shared memory,
//                       right-looking column by column, the trailing
//                       triangle spread evenly over the threads;
//   dtrsm_rows_kernel   the panel solve of the blocked path, one thread per
//                       row, L11 in shared memory, 32-column blocks;
//   dsyrk_tile_kernel   its trailing update on 64 x 64 tiles on or below the
//                       diagonal, k staged through shared memory.
#include <mutex>

#include "bl_common.cuh"
#include "launch.cuh"

namespace bl {
namespace {

constexpr int kDNb = 128;    // panel width of the blocked path
constexpr int kDTile = 64;   // trailing-update tile
constexpr int kDKc = 16;     // k staged per round of the update

// One block per matrix (or per diagonal block at (c0, c0) of a larger one
// when info_off >= 0: then matrices already failed are skipped and a failure
// is reported as info_off + its local index). The block's lower triangle sits
// packed column by column in shared memory (column k from k(2n - k + 1)/2),
// 66 KB at n = 128: three blocks share an SM and keep its FP64 pipe fed.
__device__ __forceinline__ int pk(int i, int k, int n) { return k * n - (k * (k - 1) >> 1) + (i - k); }

template <bool UP>
__global__ void __launch_bounds__(128)
dpotrf_cta_kernel(double *__restrict__ A, int n, int lda, int64_t strideA, int batch,
                  int *__restrict__ info, int info_off)
{
    extern __shared__ __align__(16) double Sd[];
    __shared__ int sh_fail;
    __shared__ double sh_rinv;
    const int64_t mat = blockIdx.x;
    if (info_off >= 0 && info[mat] != 0) return;
    double *__restrict__ Ab = A + mat * strideA;
    const int tid = threadIdx.x;
    if (tid == 0) sh_fail = 0;
    for (int j = 0; j < n; ++j)
        for (int i = j + tid; i < n; i += blockDim.x) Sd[pk(i, j, n)] = Ab[lidx<UP>(i, j, lda)];
    __syncthreads();

    for (int j = 0; j < n; ++j) {
        // one thread takes the pivot's root and reciprocal (FP64 square root
        // and division are long sequences on this GPU's slow FP64 pipe)
        if (tid == 0) {
            const double d = Sd[pk(j, j, n)];
            if (!(d > 0.0)) {
                sh_fail = j + 1;
            } else {
                const double ljj = sqrt(d);
                Sd[pk(j, j, n)] = ljj;
                sh_rinv = 1.0 / ljj;
            }
        }
        __syncthreads();
        if (sh_fail) break;  // uniform
        const double rinv = sh_rinv;
        for (int i = j + 1 + tid; i < n; i += blockDim.x) Sd[pk(i, j, n)] *= rinv;
        __syncthreads();
        // trailing lower triangle, balanced: thread pair p takes rows j+1+p
        // and n-1-p (m+1 entries together), each thread every other column
        // of both; n <= 128 leaves at most 64 pairs for the 128 threads
        {
            const int p = tid >> 1, h = tid & 1;
            const int ra = j + 1 + p, rb = n - 1 - p;
            if (ra <= rb) {
                const double *cj = Sd + pk(j, j, n) - j;  // cj[k] = element (k, j)
                const double la = cj[ra];
#pragma unroll 4
                for (int k = j + 1 + h; k <= ra; k += 2) {
                    double *e = Sd + pk(ra, k, n);
                    *e = fma(-la, cj[k], *e);
                }
                if (rb > ra) {
                    const double lb = cj[rb];
#pragma unroll 4
                    for (int k = j + 1 + h; k <= rb; k += 2) {
                        double *e = Sd + pk(rb, k, n);
                        *e = fma(-lb, cj[k], *e);
                    }
                }
            }
        }
        __syncthreads();
    }
    __syncthreads();
    for (int j = 0; j < n; ++j)
        for (int i = j + tid; i < n; i += blockDim.x) Ab[lidx<UP>(i, j, lda)] = Sd[pk(i, j, n)];
    if (tid == 0) {
        if (info_off < 0) info[mat] = sh_fail;
        else if (sh_fail) info[mat] = info_off + sh_fail;
    }
}

// L21 = A21 L11^{-T} for the rows below the diagonal block at (c0, c0): one
// thread per row, 128 rows a block; L11 (128 x 128, lower) in shared memory
// column-major; the row solved 32 columns at a time: a block first subtracts
// the row's solved blocks (read back from memory), then substitutes against
// L11's diagonal 32 x 32 block.
template <bool UP>
__global__ void __launch_bounds__(128)
dtrsm_rows_kernel(double *__restrict__ A, int n, int lda, int64_t strideA, int c0,
                  const int *__restrict__ info)
{
    extern __shared__ __align__(16) double Ld[];  // Ld[i + k * 128] = L11(i, k), i >= k
    __shared__ double rdiag[kDNb];                // 1 / L11(j, j)
    const int64_t mat = blockIdx.x;
    if (info[mat] != 0) return;
    double *__restrict__ Ab = A + mat * strideA;
    const int tid = threadIdx.x;
    for (int k = 0; k < kDNb; ++k)
        for (int i = k + tid; i < kDNb; i += blockDim.x)
            Ld[i + k * kDNb] = Ab[lidx<UP>(c0 + i, c0 + k, lda)];
    __syncthreads();
    for (int j = tid; j < kDNb; j += blockDim.x) rdiag[j] = 1.0 / Ld[j + j * kDNb];
    __syncthreads();
    const int row = c0 + kDNb + blockIdx.y * blockDim.x + tid;
    if (row >= n) return;
    double *X = Ab + lidx<UP>(row, c0, lda);  // X[k * xs] = element (row, c0 + k)
    const int64_t xs = UP ? 1 : lda;
#pragma unroll 1
    for (int jb = 0; jb < kDNb / 32; ++jb) {
        double x[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) x[c] = X[(int64_t)(32 * jb + c) * xs];
#pragma unroll 1
        for (int kk = 0; kk < 32 * jb; ++kk) {
            const double xk = X[(int64_t)kk * xs];  // solved
            const double *Lrow = Ld + 32 * jb + kk * kDNb;  // L11(32jb + c, kk)
#pragma unroll
            for (int c = 0; c < 32; ++c) x[c] = fma(-xk, Lrow[c], x[c]);
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const int j = 32 * jb + c;
            x[c] *= rdiag[j];
#pragma unroll
            for (int t = c + 1; t < 32; ++t) x[t] = fma(-x[c], Ld[32 * jb + t + j * kDNb], x[t]);
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) X[(int64_t)(32 * jb + c) * xs] = x[c];
    }
}

// A22 <- A22 - L21 L21^T on the 64 x 64 tile (I, K), I >= K, of the trailing
// lower triangle (rows/cols from c1 = c0 + 128): 256 threads, 4 x 4 outputs
// each, k staged 16 at a time.
template <bool UP>
__global__ void __launch_bounds__(256)
dsyrk_tile_kernel(double *__restrict__ A, int n, int lda, int64_t strideA, int c0,
                  const int *__restrict__ info)
{
    __shared__ double As[kDKc][kDTile + 1], Bs[kDKc][kDTile + 1];
    const int64_t mat = blockIdx.x;
    if (info[mat] != 0) return;
    int I, K;
    {
        const int t = blockIdx.y;
        int i = (int)((sqrtf(8.0f * (float)t + 1.0f) - 1.0f) * 0.5f);
        while ((i + 1) * (i + 2) / 2 <= t) ++i;
        while (i * (i + 1) / 2 > t) --i;
        I = i;
        K = t - i * (i + 1) / 2;
    }
    double *__restrict__ Ab = A + mat * strideA;
    const int c1 = c0 + kDNb, m = n - c1;
    const int ri = I * kDTile, rk = K * kDTile;
    const int tid = threadIdx.x, ty = tid & 15, tx = tid >> 4;
    double acc[4][4] = {};
#pragma unroll 1
    for (int kc = 0; kc < kDNb; kc += kDKc) {
        for (int e = tid; e < kDKc * kDTile; e += 256) {
            const int r = e % kDTile, k = e / kDTile;
            As[k][r] = ri + r < m ? Ab[lidx<UP>(c1 + ri + r, c0 + kc + k, lda)] : 0.0;
            Bs[k][r] = rk + r < m ? Ab[lidx<UP>(c1 + rk + r, c0 + kc + k, lda)] : 0.0;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kDKc; ++k) {
            double a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a[u] = As[k][ty + 16 * u];
                b[u] = Bs[k][tx + 16 * u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = fma(a[u], b[v], acc[u][v]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int gr = ri + ty + 16 * u, gc = rk + tx + 16 * v;
            if (gr < m && gc < m && gr >= gc) Ab[lidx<UP>(c1 + gr, c1 + gc, lda)] -= acc[u][v];
        }
}

template <bool UP>
int launch_dcta(double *A, int n, int lda, int64_t strideA, int batch, int *info,
                cudaStream_t st, int info_off)
{
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(dpotrf_cta_kernel<UP>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kDNb * kDNb * 8);
    });
    if (attr != cudaSuccess) return (int)attr;
    const size_t smem = (size_t)n * (n + 1) / 2 * 8;
    dpotrf_cta_kernel<UP><<<(unsigned)batch, 128, smem, st>>>(A, n, lda, strideA, batch, info,
                                                             info_off);
    return (int)cudaGetLastError();
}

template <bool UP>
int launch_dblocked(double *A, int n, int lda, int64_t strideA, int batch, int *info,
                    cudaStream_t st)
{
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(dtrsm_rows_kernel<UP>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kDNb * kDNb * 8);
    });
    if (attr != cudaSuccess) return (int)attr;
    for (int c0 = 0; c0 < n; c0 += kDNb) {
        const int nb = n - c0 < kDNb ? n - c0 : kDNb;
        int e = launch_dcta<UP>(A + c0 + (int64_t)c0 * lda, nb, lda, strideA, batch, info, st,
                                c0 == 0 ? -1 : c0);
        if (e) return e;
        const int m = n - c0 - nb;
        if (m <= 0) break;
        dim3 gt((unsigned)batch, (unsigned)((m + 127) / 128));
        dtrsm_rows_kernel<UP><<<gt, 128, kDNb * kDNb * 8, st>>>(A, n, lda, strideA, c0, info);
        if ((e = (int)cudaGetLastError())) return e;
        const int T = (m + kDTile - 1) / kDTile;
        dim3 gs((unsigned)batch, (unsigned)(T * (T + 1) / 2));
        dsyrk_tile_kernel<UP><<<gs, 256, 0, st>>>(A, n, lda, strideA, c0, info);
        if ((e = (int)cudaGetLastError())) return e;
    }
    return 0;
}

}  // namespace

int launch_dpotrf(double *A, int n, int lda, int64_t strideA, int batch, int *info,
                  cudaStream_t stream, bool upper)
{
    if (n <= kDNb)
        return upper ? launch_dcta<true>(A, n, lda, strideA, batch, info, stream, -1)
                     : launch_dcta<false>(A, n, lda, strideA, batch, info, stream, -1);
    return upper ? launch_dblocked<true>(A, n, lda, strideA, batch, info, stream)
                 : launch_dblocked<false>(A, n, lda, strideA, batch, info, stream);
}

}  // namespace bl
