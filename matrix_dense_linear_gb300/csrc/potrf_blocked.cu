// K3: batched SPOTRF for n > 128, right-looking blocked with 128-wide panels.
//
// For each panel c0 = 0, 128, 256, ... (three launches over the whole batch):
//   potf2  the 128 x 128 diagonal block A11 is factored in place by K2
//          (potrf_cta.cu) in its sub-block mode;
//   trsm   L21 = A21 L11^{-T} for the rows below it (one thread per row,
//          32-column blocks, L11 packed in shared memory);
//   syrk   A22 <- A22 - L21 L21^T on the trailing LOWER triangle only, in
//          128 x 128 tiles (only tiles on or below the diagonal are launched).
// On the tensor-core path the update is delayed by one panel where the
// trailing matrix spans more than one tile: panel p updates only panel p+1's
// columns, and panel p+1 then applies both panels' updates to the rest at once
// (k = 256), which halves the passes over the trailing matrix, the largest
// memory traffic of the schedule (n = 1024: 50 tile passes instead of 84), on
// large batches (delay_pays).
// This is the blocked right-looking schedule of "BatchLAS perf_blackwell"
// (potrf Blocked nb/W rows: nb = 128 won above n = 512) and of the blocked
// driver on "kernelbot-cholesky-930185", whose measured defect (a full-square
// trailing update costing 2n^3/3) the lower-only tiling avoids.
//
// On large batches of more than two panels the automatic route takes the
// left-looking order of the same kernels instead (launch_left, below): per
// panel its columns updated by every earlier panel at once, then its diagonal
// factor and panel solve.
//
// A matrix whose info is already nonzero after a panel is skipped by every
// later launch.
#include <mutex>

#include "bl_common.cuh"
#include "launch.cuh"

namespace bl {
namespace {

constexpr int kNb = 128;          // panel width
constexpr int kTrsmRows = 128;    // rows per TRSM block (one per thread)
constexpr int kTile = 128;        // SYRK output tile
constexpr int kKc = 16;           // SYRK k-slice staged in shared memory
constexpr int kInvMinRows = 256;  // inverse-based panel solve from two row blocks on

// L11 in shared memory, packed by 32-column blocks: block b keeps rows
// 32b .. 127 of its 32 columns, column-major with leading dimension 128 - 32b.
__host__ __device__ constexpr int l11_off(int b) { return 32 * (128 * b - 32 * (b * (b - 1) / 2)); }
constexpr int kL11Floats = l11_off(4);  // 10240 floats, 40 KB

__device__ __forceinline__ const float *l11_col(const float *Ls, int k)
{
    // pointer p with p[i] = L11(i, k) for i >= 32*(k/32)
    const int b = k >> 5;
    return Ls + l11_off(b) + (k - 32 * b) * (128 - 32 * b) - 32 * b;
}

// L21 (rows c0+128 .. n-1, columns c0 .. c0+127) <- A21 L11^{-T}, one thread
// per row (the trsm_panel kernel of "kernelbot-cholesky-930185": row in
// registers, L11 broadcast from shared memory), in four 32-column blocks:
// block jb first subtracts the row's already solved blocks kb < jb (reloaded
// from memory, the next one prefetched while the current one is applied),
// then solves against L11's diagonal block jb.
template <bool UP>
__global__ void __launch_bounds__(kTrsmRows, 3)
trsm_panel_kernel(float *__restrict__ A, int n, int lda, int64_t strideA, int c0,
                  const int *__restrict__ info)
{
    __shared__ __align__(16) float Ls[kL11Floats];
    __shared__ float rinv[kNb];
    const int64_t mat = blockIdx.x;
    if (block_skip(info, mat)) return;
    float *__restrict__ Ab = A + mat * strideA;
    const float *L11 = Ab + c0 + (int64_t)c0 * lda;  // element (c0, c0), either storage
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    for (int j = warp; j < kNb; j += kTrsmRows / 32) {
        float *dst = const_cast<float *>(l11_col(Ls, j));
        for (int i = j + lane; i < kNb; i += 32) cp_async4(dst + i, L11 + lidx<UP>(i, j, lda));
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    if (tid < kNb) rinv[tid] = 1.0f / l11_col(Ls, tid)[tid];
    __syncthreads();

    const int r0 = c0 + kNb;
    const int row = r0 + blockIdx.y * kTrsmRows + tid;
    if (row >= n) return;
    // X[k * xs] = element (row, c0 + k) of L
    float *X = Ab + lidx<UP>(row, c0, lda);
    const int64_t xs = UP ? 1 : lda;

#pragma unroll 1
    for (int jb = 0; jb < kNb / 32; ++jb) {
        float x[32], xp[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) x[c] = X[(int64_t)(32 * jb + c) * xs];
        if (jb > 0) {
#pragma unroll
            for (int c = 0; c < 32; ++c) xp[c] = X[(int64_t)c * xs];
        }
#pragma unroll 1
        for (int kb = 0; kb < jb; ++kb) {
            float xn[32];
            if (kb + 1 < jb) {
#pragma unroll
                for (int c = 0; c < 32; ++c) xn[c] = X[(int64_t)(32 * (kb + 1) + c) * xs];
            }
#pragma unroll
            for (int kk = 0; kk < 32; ++kk) {
                // L11(32jb + c, 32kb + kk), c = 0..31
                const float *Lrow = l11_col(Ls, 32 * kb + kk) + 32 * jb;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 l4 = reinterpret_cast<const float4 *>(Lrow)[q];
                    x[4 * q + 0] = fmaf(-xp[kk], l4.x, x[4 * q + 0]);
                    x[4 * q + 1] = fmaf(-xp[kk], l4.y, x[4 * q + 1]);
                    x[4 * q + 2] = fmaf(-xp[kk], l4.z, x[4 * q + 2]);
                    x[4 * q + 3] = fmaf(-xp[kk], l4.w, x[4 * q + 3]);
                }
            }
            if (kb + 1 < jb) {
#pragma unroll
                for (int c = 0; c < 32; ++c) xp[c] = xn[c];
            }
        }
        // solve against the 32 x 32 diagonal block of L11
        const float *Ld = l11_col(Ls, 32 * jb) + 32 * jb;  // Ld[c + j*ld] = L11(32jb+c, 32jb+j)
        const int ldd = 128 - 32 * jb;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            x[j] *= rinv[32 * jb + j];
            const float *Lj = Ld + j * ldd;
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
        for (int c = 0; c < 32; ++c) X[(int64_t)(32 * jb + c) * xs] = x[c];
    }
}

// A22 <- A22 - L21 L21^T on one 128 x 128 tile (I, K), I >= K, of the
// trailing lower triangle (rows/cols c1 .. n-1, c1 = c0 + 128); L21 is the
// panel's columns c0 .. c0+127. A register-tiled FP32 GEMM: 256 threads, 8 x 8
// outputs each (rows 4ty+{0..3} and 64+4ty+{0..3}, columns likewise with tx),
// the k dimension staged 16 at a time in double-buffered shared memory by
// asynchronous copies, so the next slice loads while this one is multiplied.
// The register tile follows the 128 x 128 x 8 macro tile with 8 x 8 per thread
// of "BatchLAS perf_gemm" (register_128x128 section). Only tiles on or below
// the diagonal are launched; diagonal tiles mask their upper half at the store.
__device__ __forceinline__ void syrk_stage(float (*As)[kTile + 4], float (*Bs)[kTile + 4],
                                           const float *Li, const float *Lk, int lda, int kc,
                                           int mi, int mk, bool vec, int tid)
{
    // rows [0, mi) of the I operand and [0, mk) of the K operand exist; the
    // rest of the 128 rows are zero-filled
    if (vec) {
#pragma unroll
        for (int e = 0; e < (kKc * kTile / 4) / 256; ++e) {
            const int idx = tid + 256 * e;       // float4 index in the 16 x 128 slice
            const int r = 4 * (idx & (kTile / 4 - 1)), k = idx / (kTile / 4);
            const int64_t o = (int64_t)(kc + k) * lda + r;
            const int bi = 4 * max(0, min(4, mi - r)), bk = 4 * max(0, min(4, mk - r));
            cp_async16_zfill(&As[k][r], Li + (bi ? o : 0), bi);
            cp_async16_zfill(&Bs[k][r], Lk + (bk ? o : 0), bk);
        }
    } else {
#pragma unroll 4
        for (int e = 0; e < (kKc * kTile) / 256; ++e) {
            const int idx = tid + 256 * e;
            const int r = idx & (kTile - 1), k = idx / kTile;
            const int64_t o = (int64_t)(kc + k) * lda + r;
            cp_async4_zfill(&As[k][r], Li + (r < mi ? o : 0), r < mi ? 4 : 0);
            cp_async4_zfill(&Bs[k][r], Lk + (r < mk ? o : 0), r < mk ? 4 : 0);
        }
    }
}

// Upper storage: element (r, k) of an operand is at L[k + r lda]; sixteen
// consecutive threads read one row's 16 k-values (coalesced 4-byte copies).
__device__ __forceinline__ void syrk_stage_upper(float (*As)[kTile + 4], float (*Bs)[kTile + 4],
                                                 const float *Li, const float *Lk, int lda,
                                                 int kc, int mi, int mk, int tid)
{
#pragma unroll 4
    for (int e = 0; e < (kKc * kTile) / 256; ++e) {
        const int idx = tid + 256 * e;
        const int k = idx & (kKc - 1), r = idx / kKc;
        const int64_t o = (int64_t)r * lda + kc + k;
        cp_async4_zfill(&As[k][r], Li + (r < mi ? o : 0), r < mi ? 4 : 0);
        cp_async4_zfill(&Bs[k][r], Lk + (r < mk ? o : 0), r < mk ? 4 : 0);
    }
}

template <bool UP>
__global__ void __launch_bounds__(256)
syrk_tile_kernel(float *__restrict__ A, int n, int lda, int64_t strideA, int c0,
                 const int *__restrict__ info)
{
    __shared__ __align__(16) float As[2][kKc][kTile + 4];
    __shared__ __align__(16) float Bs[2][kKc][kTile + 4];
    const int64_t mat = blockIdx.x;
    if (block_skip(info, mat)) return;
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
    const float *Li = Ab + lidx<UP>(c1 + ri, c0, lda);  // L21 rows ri.., column c0
    const float *Lk = Ab + lidx<UP>(c1 + rk, c0, lda);
    const int mi = m - ri, mk = m - rk;
    const bool vec = ((reinterpret_cast<uintptr_t>(Li) & 15) == 0) &&
                     ((reinterpret_cast<uintptr_t>(Lk) & 15) == 0) && ((lda & 3) == 0);
    const int tid = threadIdx.x;
    // ty (rows) fastest: a warp's 16 row groups of one column are contiguous
    const int ty = tid & 15, tx = tid >> 4;
    auto stage = [&](int buf, int kc) {
        if constexpr (UP) syrk_stage_upper(As[buf], Bs[buf], Li, Lk, lda, kc, mi, mk, tid);
        else syrk_stage(As[buf], Bs[buf], Li, Lk, lda, kc, mi, mk, vec, tid);
    };

    float acc[8][8];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = 0.0f;

    stage(0, 0);
    cp_async_commit();
#pragma unroll 1
    for (int c = 0; c < kNb / kKc; ++c) {
        if (c + 1 < kNb / kKc) stage((c + 1) & 1, (c + 1) * kKc);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const float(*as)[kTile + 4] = As[c & 1];
        const float(*bs)[kTile + 4] = Bs[c & 1];
#pragma unroll
        for (int k = 0; k < kKc; ++k) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&as[k][4 * ty]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&as[k][64 + 4 * ty]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&bs[k][4 * tx]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&bs[k][64 + 4 * tx]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(av[a], bv[b], acc[a][b]);
        }
        __syncthreads();
    }

    float *C = Ab + c1 + (int64_t)c1 * lda;  // element (c1, c1), either storage
    if constexpr (UP) {
        // element (gr, gc) of the trailing lower triangle at C[gc + gr lda]:
        // the four columns 4tx + b of one row are contiguous
        const bool full = ((reinterpret_cast<uintptr_t>(C) & 15) == 0) && ((lda & 3) == 0) &&
                          I != K && ri + kTile <= m && rk + kTile <= m;
#pragma unroll
        for (int ah = 0; ah < 2; ++ah)
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int gr = ri + 64 * ah + 4 * ty + a;
#pragma unroll
                for (int bh = 0; bh < 2; ++bh) {
                    const int gc0 = rk + 64 * bh + 4 * tx;
                    float *p = C + gc0 + (int64_t)gr * lda;
                    if (full) {
                        float4 v = *reinterpret_cast<float4 *>(p);
                        v.x -= acc[4 * ah + a][4 * bh + 0];
                        v.y -= acc[4 * ah + a][4 * bh + 1];
                        v.z -= acc[4 * ah + a][4 * bh + 2];
                        v.w -= acc[4 * ah + a][4 * bh + 3];
                        *reinterpret_cast<float4 *>(p) = v;
                    } else if (gr < m) {
#pragma unroll
                        for (int b = 0; b < 4; ++b)
                            if (gc0 + b < m && gr >= gc0 + b) p[b] -= acc[4 * ah + a][4 * bh + b];
                    }
                }
            }
        return;
    }
    const bool full = vec && ((reinterpret_cast<uintptr_t>(C) & 15) == 0) && I != K &&
                      ri + kTile <= m && rk + kTile <= m;
#pragma unroll
    for (int bh = 0; bh < 2; ++bh)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int gc = rk + 64 * bh + 4 * tx + b;
#pragma unroll
            for (int ah = 0; ah < 2; ++ah) {
                const int gr0 = ri + 64 * ah + 4 * ty;
                float *p = C + gr0 + (int64_t)gc * lda;
                if (full) {
                    float4 v = *reinterpret_cast<float4 *>(p);
                    v.x -= acc[4 * ah + 0][4 * bh + b];
                    v.y -= acc[4 * ah + 1][4 * bh + b];
                    v.z -= acc[4 * ah + 2][4 * bh + b];
                    v.w -= acc[4 * ah + 3][4 * bh + b];
                    *reinterpret_cast<float4 *>(p) = v;
                } else if (gc < m) {
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        const int gr = gr0 + a;
                        if (gr < m && gr >= gc) p[a] -= acc[4 * ah + a][4 * bh + b];
                    }
                }
            }
        }
}


}  // namespace

// Whether delaying a panel's trailing update pays: it halves the passes over
// the trailing matrix but puts a k = 256 update on the critical path, so it is
// taken only when the update launch covers at least eight waves of tiles (two
// per SM): measured on GB300, 4096 x 8, 2048 x 64 and 1024 x 512 gain 3-7 %,
// while one matrix of order 1024 loses 19 % and 60 of them 2 %.
static bool delay_pays(int m, int batch, int sms)
{
    const int64_t T = (m + kTile - 1) / kTile;
    return (int64_t)batch * (T * (T + 1) / 2) >= 8 * 2 * (int64_t)sms;
}

// Whether the left-looking schedule pays (the automatic route's choice for
// 16-byte-aligned batches without a workspace): its per-panel update launch covers
// batch x (row tiles of the panel) tiles with k growing by 128 a panel, so it
// wins once the first of them spans about five waves (two tiles an SM): on
// GB300, 1024 x 512 2.43 against 2.58 ms, 1024 x 1024 4.61 against 5.01,
// 1536 x 256 3.63 against 3.95, 2048 x 128 4.18 against 4.41; it loses below
// (2048 x 64 2.58 against 2.49 ms, 3072 x 16 3.09 against 2.44, one matrix of
// order 1024 0.45 against 0.33), where the longer updates sit on the panel
// chain. Two panels (n <= 256) keep the right-looking order, which fuses a
// one-tile update into the panel solve (200 x 4096: 0.65 against 0.69 ms).
bool left_pays(int n, int batch, int sms)
{
    const int64_t rows_below = (n - 1) / kTile;  // row tiles below the first panel
    return n > 2 * kTile && (int64_t)batch * rows_below >= 10 * (int64_t)sms;
}

int launch_blocked(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                   cudaStream_t stream, bool upper, float *W)
{
    // pending: the previous panel updated only this panel's columns (a narrow
    // update); its update of everything right of them is applied together with
    // this panel's, with k = 256 (both panels' columns), so that each trailing
    // tile is read and written once per two panels
    bool pending = false;
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return (int)cudaGetLastError();
    for (int c0 = 0; c0 < n; c0 += kNb) {
        const int nb = n - c0 < kNb ? n - c0 : kNb;
        int e = launch_cta(A + c0 + (int64_t)c0 * lda, nb, lda, strideA, batch, info, stream,
                           InfoMode{c0 == 0 ? -1 : c0}, upper);
        if (e) return e;
        const int m = n - c0 - nb;
        if (m <= 0) break;
        // block updates of the panel solve on the tensor cores when aligned;
        // a one-tile trailing matrix is updated by the same launch where that
        // measured faster on GB300: the upper storage (4096 matrices of order
        // 256: 1.02 against 1.10 ms), a ragged tile (order 200: 0.77 against
        // 0.80 ms) and smaller batches (64 of order 256: 63 against 67 us), but
        // not a full tile of a large batch (4096 of order 256: 0.80 either way,
        // 1 % slower fused); never while an update is pending (it takes the
        // two panels' columns)
        const bool fuse = !pending && m <= kTile && (upper || m < kTile || batch <= 2048);
        // with a workspace, panels with at least kInvMinRows rows below the
        // diagonal block are solved by its inverse (computed once, shared by
        // the panel's row blocks)
        e = 1;
        if (W != nullptr && !fuse && m >= kInvMinRows)
            e = launch_trsm_inv(A, n, lda, strideA, batch, info, c0, W, stream, upper);
        if (e == 1) e = launch_trsm_tc(A, n, lda, strideA, batch, info, c0, stream, upper, fuse);
        if (e == 0 && fuse) continue;
        if (e == 1) {
            dim3 gt((unsigned)batch, (unsigned)((m + kTrsmRows - 1) / kTrsmRows));
            if (upper)
                trsm_panel_kernel<true><<<gt, kTrsmRows, 0, stream>>>(A, n, lda, strideA, c0,
                                                                      info);
            else
                trsm_panel_kernel<false><<<gt, kTrsmRows, 0, stream>>>(A, n, lda, strideA, c0,
                                                                       info);
            e = (int)cudaGetLastError();
        }
        if (e) return e;
        // tensor cores (3xTF32) when the panels are 16-byte aligned, else FP32
        if (pending) {
            // the previous panel's delayed update and this panel's, k = 256
            e = launch_syrk_tc(A, n, lda, strideA, batch, info, c0 - kNb, 2 * kNb, false, stream,
                               upper);
            pending = false;
        } else if (m > kTile && delay_pays(m, batch, sms)) {
            // delay: only the next panel's columns now (one tile column)
            e = launch_syrk_tc(A, n, lda, strideA, batch, info, c0, kNb, true, stream, upper);
            pending = e == 0;
            if (e == 1) {  // unaligned: the FP32 kernel updates everything now
                const int T = (m + kTile - 1) / kTile;
                dim3 gs((unsigned)batch, (unsigned)(T * (T + 1) / 2));
                if (upper)
                    syrk_tile_kernel<true><<<gs, 256, 0, stream>>>(A, n, lda, strideA, c0, info);
                else
                    syrk_tile_kernel<false><<<gs, 256, 0, stream>>>(A, n, lda, strideA, c0, info);
                e = (int)cudaGetLastError();
            }
        } else {
            e = launch_syrk_tc(A, n, lda, strideA, batch, info, c0, kNb, false, stream, upper);
            if (e == 1) {
                const int T = (m + kTile - 1) / kTile;
                dim3 gs((unsigned)batch, (unsigned)(T * (T + 1) / 2));
                if (upper)
                    syrk_tile_kernel<true><<<gs, 256, 0, stream>>>(A, n, lda, strideA, c0, info);
                else
                    syrk_tile_kernel<false><<<gs, 256, 0, stream>>>(A, n, lda, strideA, c0, info);
                e = (int)cudaGetLastError();
            }
        }
        if (e) return e;
    }
    return 0;
}

// The SM count of the current device; 152 (a GB300's) when none is visible,
// so that the route query answers on a host without a GPU.
int sm_count_or_default()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0) {
        cudaGetLastError();  // no device visible: clear the error
        return 152;
    }
    return sms;
}

// The left-looking schedule of the same kernels (the automatic route's choice
// where left_pays holds, and a forced route above order 128): per panel p, its
// columns are first updated by every earlier panel at once,
// A[c0:, c0:c0+128] -= L[c0:, :c0] L[c0:c0+128, :c0]^T
// (the tensor-core update in its one-tile-column form with k = c0), then its
// diagonal block is factored and its rows below solved. Each element of the
// panel is written once per panel instead of once per earlier panel, but the
// update's k, and so its latency, grows with p. Unaligned batches take the
// right-looking driver.
int launch_left(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                cudaStream_t stream, bool upper)
{
    if (((reinterpret_cast<uintptr_t>(A) & 15) != 0) || (lda & 3) || (strideA & 3))
        return launch_blocked(A, n, lda, strideA, batch, info, stream, upper, nullptr);
    for (int c0 = 0; c0 < n; c0 += kNb) {
        const int nb = n - c0 < kNb ? n - c0 : kNb;
        int e = 0;
        if (c0 > 0 &&
            (e = launch_syrk_tc(A, n, lda, strideA, batch, info, 0, c0, true, stream, upper)))
            return e;
        if ((e = launch_cta(A + c0 + (int64_t)c0 * lda, nb, lda, strideA, batch, info, stream,
                            InfoMode{c0 == 0 ? -1 : c0}, upper)))
            return e;
        if (n - c0 - nb <= 0) break;
        if ((e = launch_trsm_tc(A, n, lda, strideA, batch, info, c0, stream, upper, false)))
            return e;
    }
    return 0;
}

int attrs_blocked(int n, cudaFuncAttributes *fa, int *threads, int *dyn_smem)
{
    // the dominant kernel of the blocked path is the trailing update (the
    // tensor-core one for aligned panels)
    (void)n;
    *threads = 256;
    *dyn_smem = 0;
    return attrs_syrk_tc(fa);
}

}  // namespace bl
