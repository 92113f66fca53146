// Batched Cholesky for 64 < n <= 128 with one warp per 32 x 32 tile of the
// lower triangle: NT = ceil(n / 32) block rows, NT(NT+1)/2 warps a matrix (6
// or 10), each lane holding one row of its tile in registers. The complex
// (CPOTRF) path runs it; T = float builds the same schedule for real input.
//
// Tile (R, C), lane l: t[k] = a(32R + l, 32C + k). Right-looking by block
// column C (a panel):
//   1. the panel's warps (tiles (R, C), R >= C) take its columns one at a
//      time: the diagonal warp publishes column j of its tile unscaled to a
//      double-buffered shared column, a barrier of the panel's warps, and every
//      lane of the panel updates its row with s = rsqrt(re d_j):
//        l = t[j] s,  t[k] -= (l s) conj(c_k)  for k > j   (= l conj(l_kj));
//   2. the tiles below the diagonal publish their finished rows of L to
//      shared memory (transposed, double-buffered by panel parity);
//   3. after a block barrier every tile right of the panel (C' > C) subtracts
//      L(R', C) L(C', C)^H from itself: a loop over the panel's 32 columns
//      that is the same for every warp and every panel, so it stays rolled;
//      the tiles of the next panel finish it before their own steps, the
//      others overlap it with those steps.
// The upper storage (U = L^H) is factored as conj(A) = A^T with the same
// steps, no conjugation (as in the n <= 64 register kernels). Rows and
// columns n .. 32 NT - 1 are an identity block. info: the lowest failing row
// of the first failing diagonal tile.
#include <mutex>

#include "bl_common.cuh"
#include "launch.cuh"

namespace bl {
namespace {

template <typename T>
struct TileOps;

template <>
struct TileOps<float> {
    static constexpr int kPerVec = 4;  // entries a 16-byte broadcast load
    __device__ static float re(float x) { return x; }
    __device__ static float zero() { return 0.0f; }
    __device__ static float one() { return 1.0f; }
    __device__ static float of_real(float r) { return r; }
    __device__ static float scale(float x, float s) { return x * s; }
    // c - a conj(b)
    __device__ static float sub_mul_conj(float c, float a, float b) { return fmaf(-a, b, c); }
    __device__ static void unpack(const float4 &v, float (&o)[4])
    {
        o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
    }
};

template <>
struct TileOps<float2> {
    static constexpr int kPerVec = 2;
    __device__ static float re(float2 x) { return x.x; }
    __device__ static float2 zero() { return make_float2(0.0f, 0.0f); }
    __device__ static float2 one() { return make_float2(1.0f, 0.0f); }
    __device__ static float2 of_real(float r) { return make_float2(r, 0.0f); }
    __device__ static float2 scale(float2 x, float s) { return make_float2(x.x * s, x.y * s); }
    __device__ static float2 sub_mul_conj(float2 c, float2 a, float2 b)
    {
        return make_float2(fmaf(-a.x, b.x, fmaf(-a.y, b.y, c.x)),
                           fmaf(-a.y, b.x, fmaf(a.x, b.y, c.y)));
    }
    __device__ static void unpack(const float4 &v, float2 (&o)[2])
    {
        o[0] = make_float2(v.x, v.y);
        o[1] = make_float2(v.z, v.w);
    }
};

template <typename T, int NT>
struct TileGeom {
    static constexpr int kWarps = NT * (NT + 1) / 2;
    static constexpr int kThreads = 32 * kWarps;
    static constexpr int kTile = 32 * 32;  // elements of one published tile
    // two shared columns, then two panel buffers of NT - 1 tiles each
    static constexpr size_t kColBytes = 2 * 32 * sizeof(T);
    static constexpr size_t kBytes = kColBytes + 2 * (size_t)(NT - 1) * kTile * sizeof(T);
};

// warp w -> tile (R, C), enumerated column by column: (0,0), (1,0), .., (NT-1,0), (1,1), ..
template <int NT>
__device__ __forceinline__ void tile_of(int w, int &R, int &C)
{
    int c = 0, first = 0;
#pragma unroll
    for (int q = 0; q < NT; ++q) {
        const int cnt = NT - q;  // tiles of column q
        if (c == q && w >= first + cnt) {
            first += cnt;
            c = q + 1;
        }
    }
    C = c;
    R = c + (w - first);
}

// real: three blocks an SM (64 registers at NT = 4, no spill; 1024 matrices of
// order 127 70.8 against 74.9 us at two blocks, 4096 of order 112 221 against
// 254 us); complex: two (96 registers)
template <typename T, int NT, bool UP>
__global__ void __launch_bounds__(TileGeom<T, NT>::kThreads, sizeof(T) == 4 ? 3 : 2)
potrf_tiles_kernel(T *__restrict__ A, int n, int lda, int64_t strideA, int batch,
                   int *__restrict__ info, int info_off)
{
    using X = TileOps<T>;
    using Gm = TileGeom<T, NT>;
    constexpr int V = X::kPerVec;
    extern __shared__ __align__(16) uint8_t sraw[];
    T *col = reinterpret_cast<T *>(sraw);                      // [2][32]
    T *panel = reinterpret_cast<T *>(sraw + Gm::kColBytes);    // [2][NT-1][32 k][32 l]
    __shared__ unsigned bad_rows[NT];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int R, Cw;
    tile_of<NT>(warp, R, Cw);
    const int64_t mat = blockIdx.x;  // the grid is the batch
    T *__restrict__ Ab = A + mat * strideA;
    const int row = 32 * R + lane;
    const bool live = row < n;
    const bool diag = R == Cw;
    pdl_wait();
    pdl_trigger();
    // a diagonal block of a larger matrix (info_off >= 0): skip a matrix that
    // failed in an earlier block (one block per matrix: the read is uniform)
    if (info_off >= 0 && info[mat] != 0) return;

    T t[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) t[k] = (diag && k == lane) ? X::one() : X::zero();
#pragma unroll
    for (int k = 0; k < 32; ++k)
        if (live && (!diag || k <= lane)) t[k] = Ab[lidx<UP>(row, 32 * Cw + k, lda)];

    float dm = 1.0f;  // a diagonal lane's pivot
    for (int C = 0; C < NT; ++C) {
        if (Cw == C) {
            const int steps = n - 32 * C < 32 ? n - 32 * C : 32;
            const int nthreads = 32 * (NT - C);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (j >= steps) break;  // uniform over the panel's warps
                T *cb = col + 32 * (j & 1);
                if (diag) cb[lane] = t[j];
                named_bar_sync(1, nthreads);
                const float d = X::re(cb[j]);
                const float s = rsqrt_approx(d);
                const T l = X::scale(t[j], s);
                const T w = X::scale(l, s);
                t[j] = l;
                dm = (diag && lane == j) ? d : dm;
#pragma unroll
                for (int q = (j + 1) / V; q < 32 / V; ++q) {
                    T cv[V];
                    X::unpack(reinterpret_cast<const float4 *>(cb)[q], cv);
#pragma unroll
                    for (int u = 0; u < V; ++u) {
                        const int k = V * q + u;
                        if (k > j) t[k] = X::sub_mul_conj(t[k], w, cv[u]);
                    }
                }
            }
            if (!diag) {  // publish this row of L(R, C), transposed
                T *P = panel + ((size_t)(C & 1) * (NT - 1) + (R - C - 1)) * Gm::kTile;
#pragma unroll
                for (int k = 0; k < 32; ++k) P[32 * k + lane] = t[k];
            } else {
                const unsigned bad = __ballot_sync(0xffffffffu, live && !pivot_ok(dm));
                if (lane == 0) bad_rows[C] = bad;
            }
        }
        __syncthreads();
        if (Cw > C) {  // A(R, Cw) -= L(R, C) L(Cw, C)^H
            const T *Pa = panel + ((size_t)(C & 1) * (NT - 1) + (R - C - 1)) * Gm::kTile;
            const T *Pb = panel + ((size_t)(C & 1) * (NT - 1) + (Cw - C - 1)) * Gm::kTile;
#pragma unroll 1
            for (int k = 0; k < 32; ++k) {
                const T a = Pa[32 * k + lane];
                const float4 *lb = reinterpret_cast<const float4 *>(Pb + 32 * k);
#pragma unroll
                for (int q = 0; q < 32 / V; ++q) {
                    T cv[V];
                    X::unpack(lb[q], cv);
#pragma unroll
                    for (int u = 0; u < V; ++u)
                        t[V * q + u] = X::sub_mul_conj(t[V * q + u], a, cv[u]);
                }
            }
        }
    }

    asm volatile("" : "+r"(lda));  // no load address lives to the stores
#pragma unroll
    for (int k = 0; k < 32; ++k)
        if (live && (!diag || k < lane)) Ab[lidx<UP>(row, 32 * Cw + k, lda)] = t[k];
    if (diag && live) Ab[lidx<UP>(row, row, lda)] = X::of_real(sqrt_approx(dm));
    __syncthreads();
    if (threadIdx.x == 0) {
        int f = 0;
        for (int C = 0; C < NT && !f; ++C)
            if (bad_rows[C]) f = 32 * C + __ffs(bad_rows[C]);
        if (info_off < 0) info[mat] = f;
        else if (f) info[mat] = info_off + f;
    }
}

template <typename T, int NT, bool UP>
int launch_t(T *A, int n, int lda, int64_t strideA, int batch, int *info, cudaStream_t st,
             int info_off)
{
    using Gm = TileGeom<T, NT>;
    static DeviceOnce attrs;
    if (const int e = attrs.run([] {
            return cudaFuncSetAttribute(potrf_tiles_kernel<T, NT, UP>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)Gm::kBytes);
        }))
        return e;
    return launch_pdl(potrf_tiles_kernel<T, NT, UP>, dim3((unsigned)batch), dim3(Gm::kThreads),
                      Gm::kBytes, st, A, n, lda, strideA, batch, info, info_off);
}

template <typename T>
int launch_tiles(T *A, int n, int lda, int64_t strideA, int batch, int *info, cudaStream_t st,
                 bool upper, int info_off)
{
    if (n <= 64 || n > 128) return -1;
    if (n <= 96)
        return upper ? launch_t<T, 3, true>(A, n, lda, strideA, batch, info, st, info_off)
                     : launch_t<T, 3, false>(A, n, lda, strideA, batch, info, st, info_off);
    return upper ? launch_t<T, 4, true>(A, n, lda, strideA, batch, info, st, info_off)
                 : launch_t<T, 4, false>(A, n, lda, strideA, batch, info, st, info_off);
}

}  // namespace

int launch_cpotrf_tiles(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                        cudaStream_t stream, bool upper, int info_off)
{
    return launch_tiles(reinterpret_cast<float2 *>(A), n, lda, strideA, batch, info, stream,
                        upper, info_off);
}

int launch_spotrf_tiles(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                        cudaStream_t stream, bool upper, int info_off)
{
    return launch_tiles(A, n, lda, strideA, batch, info, stream, upper, info_off);
}

int attrs_tiles(int n, cudaFuncAttributes *fa, int *threads, int *dyn_smem)
{
    if (n <= 96) {
        *threads = TileGeom<float, 3>::kThreads;
        *dyn_smem = (int)TileGeom<float, 3>::kBytes;
        return (int)cudaFuncGetAttributes(fa, potrf_tiles_kernel<float, 3, false>);
    }
    *threads = TileGeom<float, 4>::kThreads;
    *dyn_smem = (int)TileGeom<float, 4>::kBytes;
    return (int)cudaFuncGetAttributes(fa, potrf_tiles_kernel<float, 4, false>);
}

}  // namespace bl
