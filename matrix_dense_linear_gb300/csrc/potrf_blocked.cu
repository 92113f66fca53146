// K3: batched SPOTRF for n > 128, right-looking blocked with 128-wide panels.
//
// For each panel c0 = 0, 128, 256, ... (three launches over the whole batch):
//   potf2  the 128 x 128 diagonal block A11 is factored in place by K2
//          (potrf_cta.cu) in its sub-block mode;
//   trsm   L21 = A21 L11^{-T} for the rows below it (one thread per row,
//          32-column blocks, L11 staged in shared memory);
//   syrk   A22 <- A22 - L21 L21^T on the trailing LOWER triangle only, in
//          64 x 64 tiles (only tiles on or below the diagonal are launched).
// This is the blocked right-looking schedule of "BatchLAS perf_blackwell"
// (potrf Blocked nb/W rows: nb = 128 won above n = 512) and of the blocked
// driver on "kernelbot-cholesky-930185", whose measured defect (a full-square
// trailing update costing 2n^3/3) the lower-only tiling avoids.
//
// A matrix whose info is already nonzero after a panel is skipped by every
// later launch.
#include <mutex>

#include "bl_common.cuh"

namespace bl {
namespace {

constexpr int kNb = 128;          // panel width
constexpr int kTrsmRows = 128;    // rows per TRSM block (one per thread)
constexpr int kLdL = kNb + 4;     // shared leading dimension of L11
constexpr int kTile = 64;         // SYRK output tile
constexpr int kKc = 32;           // SYRK k-chunk staged in shared memory

// L21 (rows c0+128 .. n-1, columns c0 .. c0+127) <- A21 L11^{-T}.
__global__ void __launch_bounds__(kTrsmRows)
trsm_panel_kernel(float *__restrict__ A, int n, int lda, int64_t strideA, int c0,
                  const int *__restrict__ info)
{
    extern __shared__ __align__(16) float Ls[];  // [kNb][kLdL]: Ls[i + j*kLdL] = L11(i, j)
    __shared__ float rinv[kNb];
    const int64_t mat = blockIdx.x;
    if (info[mat] != 0) return;
    float *__restrict__ Ab = A + mat * strideA;
    const float *L11 = Ab + c0 + (int64_t)c0 * lda;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    for (int j = warp; j < kNb; j += kTrsmRows / 32)
        for (int i = j + lane; i < kNb; i += 32) Ls[i + j * kLdL] = L11[i + (int64_t)j * lda];
    __syncthreads();
    if (tid < kNb) rinv[tid] = 1.0f / Ls[tid + tid * kLdL];
    __syncthreads();

    const int r0 = c0 + kNb;
    const int row = r0 + blockIdx.y * kTrsmRows + tid;
    if (row >= n) return;
    float *X = Ab + row + (int64_t)c0 * lda;  // X[k*lda] = element (row, c0 + k)

#pragma unroll 1
    for (int jb = 0; jb < kNb / 32; ++jb) {
        float x[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) x[c] = X[(int64_t)(32 * jb + c) * lda];
        // subtract the solved columns 0 .. 32*jb-1
#pragma unroll 1
        for (int k = 0; k < 32 * jb; ++k) {
            const float xk = X[(int64_t)k * lda];
            const float *Lrow = Ls + 32 * jb + k * kLdL;  // L11(32jb + c, k), c = 0..31
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 l4 = reinterpret_cast<const float4 *>(Lrow)[q];
                x[4 * q + 0] = fmaf(-xk, l4.x, x[4 * q + 0]);
                x[4 * q + 1] = fmaf(-xk, l4.y, x[4 * q + 1]);
                x[4 * q + 2] = fmaf(-xk, l4.z, x[4 * q + 2]);
                x[4 * q + 3] = fmaf(-xk, l4.w, x[4 * q + 3]);
            }
        }
        // solve against the 32 x 32 diagonal block of L11
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            x[j] *= rinv[32 * jb + j];
            const float *Lj = Ls + 32 * jb + (32 * jb + j) * kLdL;
#pragma unroll
            for (int q = (j + 1) / 4; q < 8; ++q) {
                const float4 l4 = reinterpret_cast<const float4 *>(Lj)[q];
                const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int c = 4 * q + t;
                    if (c > j) x[c] = fmaf(-x[j], lv[t], x[c]);
                }
            }
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) X[(int64_t)(32 * jb + c) * lda] = x[c];
    }
}

// A22 <- A22 - L21 L21^T on one 64 x 64 tile (I, K), I >= K, of the trailing
// lower triangle (rows/cols c1 .. n-1, c1 = c0 + 128); L21 = columns c0.. .
__global__ void __launch_bounds__(256)
syrk_tile_kernel(float *__restrict__ A, int n, int lda, int64_t strideA, int c0,
                 const int *__restrict__ info)
{
    __shared__ __align__(16) float As[kKc][kTile + 4];
    __shared__ __align__(16) float Bs[kKc][kTile + 4];
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
    float *__restrict__ Ab = A + mat * strideA;
    const int c1 = c0 + kNb;
    const int m = n - c1;
    const int ri = I * kTile, rk = K * kTile;  // tile origin, trailing coordinates
    const float *Li = Ab + c1 + ri + (int64_t)c0 * lda;  // L21 rows ri.., column c0
    const float *Lk = Ab + c1 + rk + (int64_t)c0 * lda;
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;  // 16 x 16 threads, 4 x 4 each

    float acc[4][4] = {};
#pragma unroll 1
    for (int kc = 0; kc < kNb; kc += kKc) {
        // stage L21[ri .. ri+63, kc .. kc+31] and L21[rk .., ..]: 2048 floats each
#pragma unroll
        for (int e = 0; e < (kKc * kTile) / 256; ++e) {
            const int idx = tid + 256 * e;
            const int r = idx & (kTile - 1), k = idx >> 6;
            const int64_t o = (int64_t)(kc + k) * lda + r;
            As[k][r] = (ri + r < m) ? Li[o] : 0.0f;
            Bs[k][r] = (rk + r < m) ? Lk[o] : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < kKc; ++k) {
            const float4 a4 = *reinterpret_cast<const float4 *>(&As[k][4 * ty]);
            const float4 b4 = *reinterpret_cast<const float4 *>(&Bs[k][4 * tx]);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
            const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(av[a], bv[b], acc[a][b]);
        }
        __syncthreads();
    }
    float *C = Ab + c1 + (int64_t)c1 * lda;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int gc = rk + 4 * tx + b;
        if (gc >= m) continue;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int gr = ri + 4 * ty + a;
            if (gr < m && gr >= gc) {
                float *p = C + gr + (int64_t)gc * lda;
                *p = *p - acc[a][b];
            }
        }
    }
}

std::once_flag g_trsm_once;
cudaError_t g_trsm_attr = cudaSuccess;
constexpr int kTrsmSmem = kNb * kLdL * 4;

}  // namespace

int launch_blocked(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                   cudaStream_t stream)
{
    std::call_once(g_trsm_once, [] {
        g_trsm_attr = cudaFuncSetAttribute(trsm_panel_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kTrsmSmem);
    });
    if (g_trsm_attr != cudaSuccess) return (int)g_trsm_attr;
    for (int c0 = 0; c0 < n; c0 += kNb) {
        const int nb = n - c0 < kNb ? n - c0 : kNb;
        int e = launch_cta(A + c0 + (int64_t)c0 * lda, nb, lda, strideA, batch, info, stream,
                           InfoMode{c0 == 0 ? -1 : c0});
        if (e) return e;
        const int m = n - c0 - nb;
        if (m <= 0) break;
        dim3 gt((unsigned)batch, (unsigned)((m + kTrsmRows - 1) / kTrsmRows));
        trsm_panel_kernel<<<gt, kTrsmRows, kTrsmSmem, stream>>>(A, n, lda, strideA, c0, info);
        if ((e = (int)cudaGetLastError())) return e;
        const int T = (m + kTile - 1) / kTile;
        dim3 gs((unsigned)batch, (unsigned)(T * (T + 1) / 2));
        syrk_tile_kernel<<<gs, 256, 0, stream>>>(A, n, lda, strideA, c0, info);
        if ((e = (int)cudaGetLastError())) return e;
    }
    return 0;
}

int attrs_blocked(int n, cudaFuncAttributes *fa, int *threads, int *dyn_smem)
{
    // the dominant kernel of the blocked path is the trailing update
    (void)n;
    *threads = 256;
    *dyn_smem = 0;
    return (int)cudaFuncGetAttributes(fa, syrk_tile_kernel);
}

}  // namespace bl
