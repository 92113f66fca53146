// DPOTRF, CPOTRF and ZPOTRF: batched Cholesky of double-precision real and
// single- and double-precision complex (Hermitian) batches, the operation of the
// single-precision path (A = L L^T, or L L^H for complex; the upper storage
// A = U^H U; info = first pivot with !(d > 0)). "BatchLAS perf_blackwell"
// lists double and the complex types among the types of its batched potrf
// (the type columns of its potrf rows).
//
// On this GPU the FP64 pipe runs at about 1/70 of the FP32 rate (the
// library's FMA probe: 1.05 against 74.7 TFLOP/s), so a double factorization
// is bound by its FMA count; the complex one is the same algorithm with
// complex FMAs (four real ones each) on the FP32 pipes. The kernels are the
// plain forms, one element type T (double, float2 or double2: complex float
// or double) through
// the small set of operations in Ar<T>, each doing only the FMAs of the lower
// triangle, with IEEE square root and division:
//   simple_potrf_kernel n <= 128 (and the 128 x 128 diagonal blocks of larger
//                       n): the block's lower triangle in shared memory,
//                       right-looking column by column, the trailing
//                       triangle spread evenly over the threads;
//   simple_trsm_kernel  the panel solve of the blocked path, one thread per
//                       row, L11 packed in shared memory, 32-column blocks
//                       (16 for complex);
//   simple_syrk_kernel  its trailing update on 64 x 64 tiles on or below the
//                       diagonal, k staged through shared memory.
// Single-precision complex batches with 16-byte-aligned panels (either
// storage) take the tensor-core forms of the panel solve and the trailing
// update instead (ctrsm_tc.cu, cherk_tc.cu), and their diagonal blocks above
// order 64 the warp-per-tile register kernel (potrf_tiles.cu).
#include <mutex>
#include <type_traits>

#include "bl_common.cuh"
#include "launch.cuh"

namespace bl {
namespace {

// The element operations. R is the real type of the pivots; "conj" is the
// identity for real T. The upper storage keeps U = L^H, so an element of L is
// loaded and stored conjugated there.
template <typename T>
struct Ar;

template <>
struct Ar<double> {
    using R = double;
    __device__ static R re(double x) { return x; }
    __device__ static double of_real(R r) { return r; }
    __device__ static double zero() { return 0.0; }
    __device__ static double load(const double *p, bool) { return *p; }
    __device__ static void store(double *p, double v, bool) { *p = v; }
    __device__ static double scale(double x, R s) { return x * s; }
    __device__ static double sub_mul_conj(double c, double a, double b) { return fma(-a, b, c); }
    __device__ static double add_mul_conj(double c, double a, double b) { return fma(a, b, c); }
    __device__ static double sub(double c, double a) { return c - a; }
    __device__ static R root(R d) { return sqrt(d); }
    __device__ static bool pivot_pass(R d) { return d > 0.0; }
};

template <>
struct Ar<float2> {
    using R = float;
    __device__ static R re(float2 x) { return x.x; }
    __device__ static float2 of_real(R r) { return make_float2(r, 0.0f); }
    __device__ static float2 zero() { return make_float2(0.0f, 0.0f); }
    __device__ static float2 cj(float2 x) { return make_float2(x.x, -x.y); }
    __device__ static float2 load(const float2 *p, bool up) { return up ? cj(*p) : *p; }
    __device__ static void store(float2 *p, float2 v, bool up) { *p = up ? cj(v) : v; }
    __device__ static float2 scale(float2 x, R s) { return make_float2(x.x * s, x.y * s); }
    // c - a conj(b)
    __device__ static float2 sub_mul_conj(float2 c, float2 a, float2 b)
    {
        return make_float2(fmaf(-a.x, b.x, fmaf(-a.y, b.y, c.x)),
                           fmaf(-a.y, b.x, fmaf(a.x, b.y, c.y)));
    }
    // c + a conj(b)
    __device__ static float2 add_mul_conj(float2 c, float2 a, float2 b)
    {
        return make_float2(fmaf(a.x, b.x, fmaf(a.y, b.y, c.x)), fmaf(a.y, b.x, fmaf(-a.x, b.y, c.y)));
    }
    __device__ static float2 sub(float2 c, float2 a) { return make_float2(c.x - a.x, c.y - a.y); }
    __device__ static R root(R d) { return sqrtf(d); }
    // single precision: a subnormal pivot fails, as in every float kernel
    __device__ static bool pivot_pass(R d) { return pivot_ok(d); }
};

template <>
struct Ar<double2> {
    using R = double;
    __device__ static R re(double2 x) { return x.x; }
    __device__ static double2 of_real(R r) { return make_double2(r, 0.0); }
    __device__ static double2 zero() { return make_double2(0.0, 0.0); }
    __device__ static double2 cj(double2 x) { return make_double2(x.x, -x.y); }
    __device__ static double2 load(const double2 *p, bool up) { return up ? cj(*p) : *p; }
    __device__ static void store(double2 *p, double2 v, bool up) { *p = up ? cj(v) : v; }
    __device__ static double2 scale(double2 x, R s) { return make_double2(x.x * s, x.y * s); }
    __device__ static double2 sub_mul_conj(double2 c, double2 a, double2 b)
    {
        return make_double2(fma(-a.x, b.x, fma(-a.y, b.y, c.x)), fma(-a.y, b.x, fma(a.x, b.y, c.y)));
    }
    __device__ static double2 add_mul_conj(double2 c, double2 a, double2 b)
    {
        return make_double2(fma(a.x, b.x, fma(a.y, b.y, c.x)), fma(a.y, b.x, fma(-a.x, b.y, c.y)));
    }
    __device__ static double2 sub(double2 c, double2 a) { return make_double2(c.x - a.x, c.y - a.y); }
    __device__ static R root(R d) { return sqrt(d); }
    __device__ static bool pivot_pass(R d) { return d > 0.0; }
};

constexpr int kDNb = 128;    // panel width of the blocked path
constexpr int kDTile = 64;   // trailing-update tile
constexpr int kDKc = 16;     // k staged per round of the update

// One block per matrix (or per diagonal block at (c0, c0) of a larger one
// when info_off >= 0: then matrices already failed are skipped and a failure
// is reported as info_off + its local index). The block's lower triangle sits
// packed column by column in shared memory (column k from k(2n - k + 1)/2),
// 66 KB at n = 128: three blocks share an SM and keep its FP64 pipe fed.
__device__ __forceinline__ int pk(int i, int k, int n) { return k * n - (k * (k - 1) >> 1) + (i - k); }

constexpr int kPotrfThreads = 256;

template <typename T, bool UP>
__global__ void __launch_bounds__(kPotrfThreads)
simple_potrf_kernel(T *__restrict__ A, int n, int lda, int64_t strideA, int batch,
                  int *__restrict__ info, int info_off)
{
    using X = Ar<T>;
    using R = typename X::R;
    extern __shared__ __align__(16) uint8_t sraw[];
    T *Sd = reinterpret_cast<T *>(sraw);
    __shared__ int sh_fail;
    __shared__ R sh_rinv;
    const int64_t mat = blockIdx.x;
    if (info_off >= 0 && info[mat] != 0) return;
    T *__restrict__ Ab = A + mat * strideA;
    const int tid = threadIdx.x;
    if (tid == 0) sh_fail = 0;
    for (int j = 0; j < n; ++j)
        for (int i = j + tid; i < n; i += blockDim.x)
            Sd[pk(i, j, n)] = X::load(Ab + lidx<UP>(i, j, lda), UP);
    __syncthreads();

    for (int j = 0; j < n; ++j) {
        // one thread takes the pivot's root and reciprocal (FP64 square root
        // and division are long sequences on this GPU's slow FP64 pipe)
        if (tid == 0) {
            const R d = X::re(Sd[pk(j, j, n)]);  // a complex diagonal's imaginary part is not read
            if (!X::pivot_pass(d)) {
                sh_fail = j + 1;
            } else {
                const R ljj = X::root(d);
                Sd[pk(j, j, n)] = X::of_real(ljj);
                sh_rinv = R(1) / ljj;
            }
        }
        __syncthreads();
        if (sh_fail) break;  // uniform
        const R rinv = sh_rinv;
        for (int i = j + 1 + tid; i < n; i += blockDim.x)
            Sd[pk(i, j, n)] = X::scale(Sd[pk(i, j, n)], rinv);
        __syncthreads();
        // trailing lower triangle, balanced: row pair p (rows j+1+p and
        // n-1-p, m+1 entries together) goes to four threads, each taking every
        // fourth column of both; the block has 2n threads (at most 64 pairs)
        {
            const int p = tid >> 2, h = tid & 3;
            const int ra = j + 1 + p, rb = n - 1 - p;
            if (ra <= rb) {
                const T *cj = Sd + pk(j, j, n) - j;  // cj[k] = element (k, j)
                const T la = cj[ra];
#pragma unroll 4
                for (int k = j + 1 + h; k <= ra; k += 4) {  // a_(ra,k) -= l_(ra,j) conj(l_(k,j))
                    T *e = Sd + pk(ra, k, n);
                    *e = X::sub_mul_conj(*e, la, cj[k]);
                }
                if (rb > ra) {
                    const T lb = cj[rb];
#pragma unroll 4
                    for (int k = j + 1 + h; k <= rb; k += 4) {
                        T *e = Sd + pk(rb, k, n);
                        *e = X::sub_mul_conj(*e, lb, cj[k]);
                    }
                }
            }
        }
        __syncthreads();
    }
    __syncthreads();
    for (int j = 0; j < n; ++j)
        for (int i = j + tid; i < n; i += blockDim.x)
            X::store(Ab + lidx<UP>(i, j, lda), Sd[pk(i, j, n)], UP);
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
template <typename T, bool UP>
__global__ void __launch_bounds__(128)
simple_trsm_kernel(T *__restrict__ A, int n, int lda, int64_t strideA, int c0,
                  const int *__restrict__ info)
{
    using X = Ar<T>;
    using R = typename X::R;
    extern __shared__ __align__(16) uint8_t sraw[];
    T *Ld = reinterpret_cast<T *>(sraw);  // Ld[pk(i, k, 128)] = L11(i, k), i >= k (packed)
    __shared__ R rdiag[kDNb];             // 1 / L11(j, j)
    const int64_t mat = blockIdx.x;
    if (block_skip(info, mat)) return;
    T *__restrict__ Ab = A + mat * strideA;
    const int tid = threadIdx.x;
    for (int k = 0; k < kDNb; ++k)
        for (int i = k + tid; i < kDNb; i += blockDim.x)
            Ld[pk(i, k, kDNb)] = X::load(Ab + lidx<UP>(c0 + i, c0 + k, lda), UP);
    __syncthreads();
    for (int j = tid; j < kDNb; j += blockDim.x) rdiag[j] = R(1) / X::re(Ld[pk(j, j, kDNb)]);
    __syncthreads();
    const int row = c0 + kDNb + blockIdx.y * blockDim.x + tid;
    if (row >= n) return;
    // x L11^H = a, row by row: x_c = (a_c - sum_{k<c} x_k conj(l_ck)) / l_cc,
    // W columns at a time (16 for complex T, which keeps x in registers)
    constexpr int W = std::is_same<T, double>::value ? 32 : 16;  // complex: 16
    T *Xr = Ab + lidx<UP>(row, c0, lda);  // Xr[k * xs] = element (row, c0 + k)
    const int64_t xs = UP ? 1 : lda;
#pragma unroll 1
    for (int jb = 0; jb < kDNb / W; ++jb) {
        T x[W];
#pragma unroll
        for (int c = 0; c < W; ++c) x[c] = X::load(Xr + (int64_t)(W * jb + c) * xs, UP);
#pragma unroll 1
        for (int kk = 0; kk < W * jb; ++kk) {
            const T xk = X::load(Xr + (int64_t)kk * xs, UP);  // solved
            const T *Lrow = Ld + pk(W * jb, kk, kDNb);        // Lrow[c] = L11(W jb + c, kk)
#pragma unroll
            for (int c = 0; c < W; ++c) x[c] = X::sub_mul_conj(x[c], xk, Lrow[c]);
        }
#pragma unroll
        for (int c = 0; c < W; ++c) {
            const int j = W * jb + c;
            x[c] = X::scale(x[c], rdiag[j]);
#pragma unroll
            for (int t = c + 1; t < W; ++t)
                x[t] = X::sub_mul_conj(x[t], x[c], Ld[pk(W * jb + t, j, kDNb)]);
        }
#pragma unroll
        for (int c = 0; c < W; ++c) X::store(Xr + (int64_t)(W * jb + c) * xs, x[c], UP);
    }
}

// A22 <- A22 - L21 L21^T on the 64 x 64 tile (I, K), I >= K, of the trailing
// lower triangle (rows/cols from c1 = c0 + 128): 256 threads, 4 x 4 outputs
// each, k staged 16 at a time.
template <typename T, bool UP>
__global__ void __launch_bounds__(256)
simple_syrk_kernel(T *__restrict__ A, int n, int lda, int64_t strideA, int c0,
                  const int *__restrict__ info)
{
    using X = Ar<T>;
    __shared__ T As[kDKc][kDTile + 1], Bs[kDKc][kDTile + 1];
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
    T *__restrict__ Ab = A + mat * strideA;
    const int c1 = c0 + kDNb, m = n - c1;
    const int ri = I * kDTile, rk = K * kDTile;
    const int tid = threadIdx.x, ty = tid & 15, tx = tid >> 4;
    T acc[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = X::zero();
#pragma unroll 1
    for (int kc = 0; kc < kDNb; kc += kDKc) {
        for (int e = tid; e < kDKc * kDTile; e += 256) {
            const int r = e % kDTile, k = e / kDTile;
            As[k][r] = ri + r < m ? X::load(Ab + lidx<UP>(c1 + ri + r, c0 + kc + k, lda), UP)
                                  : X::zero();
            Bs[k][r] = rk + r < m ? X::load(Ab + lidx<UP>(c1 + rk + r, c0 + kc + k, lda), UP)
                                  : X::zero();
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kDKc; ++k) {
            T a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a[u] = As[k][ty + 16 * u];
                b[u] = Bs[k][tx + 16 * u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = X::add_mul_conj(acc[u][v], a[u], b[v]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int gr = ri + ty + 16 * u, gc = rk + tx + 16 * v;
            if (gr < m && gc < m && gr >= gc) {
                T *p = Ab + lidx<UP>(c1 + gr, c1 + gc, lda);
                X::store(p, X::sub(X::load(p, UP), acc[u][v]), UP);
            }
        }
}

template <typename T, bool UP>
int launch_cta_s(T *A, int n, int lda, int64_t strideA, int batch, int *info, cudaStream_t st,
                 int info_off)
{
    static DeviceOnce attrs;
    if (const int e = attrs.run([] {
            return cudaFuncSetAttribute(simple_potrf_kernel<T, UP>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)(kDNb * (kDNb + 1) / 2 * sizeof(T)));
        }))
        return e;
    const size_t smem = (size_t)n * (n + 1) / 2 * sizeof(T);
    // four threads a row pair: 2n threads (a multiple of 32, at most 256)
    const int threads = 2 * n < 32 ? 32 : ((2 * n + 31) / 32) * 32;
    simple_potrf_kernel<T, UP><<<(unsigned)batch, threads > kPotrfThreads ? kPotrfThreads : threads,
                                 smem, st>>>(A, n, lda, strideA, batch, info, info_off);
    return (int)cudaGetLastError();
}

template <typename T, bool UP>
int launch_blocked_s(T *A, int n, int lda, int64_t strideA, int batch, int *info,
                     cudaStream_t st)
{
    static DeviceOnce attrs;
    if (const int e = attrs.run([] {
            return cudaFuncSetAttribute(simple_trsm_kernel<T, UP>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)(kDNb * (kDNb + 1) / 2 * sizeof(T)));
        }))
        return e;
    for (int c0 = 0; c0 < n; c0 += kDNb) {
        const int nb = n - c0 < kDNb ? n - c0 : kDNb;
        // single-precision complex diagonal blocks above 64 on the warp-per-tile
        // register kernel (potrf_tiles.cu, complex arithmetic), the others on
        // the plain shared-memory kernel
        int e;
        if constexpr (std::is_same<T, float2>::value) {
            if (nb > 64)
                e = launch_cpotrf_tiles(reinterpret_cast<float *>(A + c0 + (int64_t)c0 * lda), nb,
                                        lda, strideA, batch, info, st, UP, c0 == 0 ? -1 : c0);
            else
                e = launch_cta_s<T, UP>(A + c0 + (int64_t)c0 * lda, nb, lda, strideA, batch,
                                        info, st, c0 == 0 ? -1 : c0);
        } else {
            e = launch_cta_s<T, UP>(A + c0 + (int64_t)c0 * lda, nb, lda, strideA, batch, info, st,
                                    c0 == 0 ? -1 : c0);
        }
        if (e) return e;
        const int m = n - c0 - nb;
        if (m <= 0) break;
        // single-precision complex, 16-byte aligned: the panel solve's block
        // updates on the tensor cores (ctrsm_tc.cu); else the FP32 kernel
        e = 1;
        if constexpr (std::is_same<T, float2>::value) {
            e = launch_ctrsm_tc(reinterpret_cast<float *>(A), n, lda, strideA, batch, info, c0,
                                st, UP);
            if (e != 0 && e != 1) return e;
        }
        if (e == 1) {
            dim3 gt((unsigned)batch, (unsigned)((m + 127) / 128));
            simple_trsm_kernel<T, UP><<<gt, 128, kDNb * (kDNb + 1) / 2 * sizeof(T), st>>>(
                A, n, lda, strideA, c0, info);
            if ((e = (int)cudaGetLastError())) return e;
        }
        // single-precision complex, 16-byte aligned: the trailing update on the
        // tensor cores (cherk_tc.cu); else the FP32 tiles below
        if constexpr (std::is_same<T, float2>::value) {
            e = launch_cherk_tc(reinterpret_cast<float *>(A), n, lda, strideA, batch, info, c0,
                                st, UP);
            if (e == 0) continue;
            if (e != 1) return e;
        }
        const int Tn = (m + kDTile - 1) / kDTile;
        dim3 gs((unsigned)batch, (unsigned)(Tn * (Tn + 1) / 2));
        simple_syrk_kernel<T, UP><<<gs, 256, 0, st>>>(A, n, lda, strideA, c0, info);
        if ((e = (int)cudaGetLastError())) return e;
    }
    return 0;
}

template <typename T>
int launch_simple(T *A, int n, int lda, int64_t strideA, int batch, int *info,
                  cudaStream_t stream, bool upper)
{
    if (n <= kDNb)
        return upper ? launch_cta_s<T, true>(A, n, lda, strideA, batch, info, stream, -1)
                     : launch_cta_s<T, false>(A, n, lda, strideA, batch, info, stream, -1);
    return upper ? launch_blocked_s<T, true>(A, n, lda, strideA, batch, info, stream)
                 : launch_blocked_s<T, false>(A, n, lda, strideA, batch, info, stream);
}

}  // namespace

int launch_dpotrf(double *A, int n, int lda, int64_t strideA, int batch, int *info,
                  cudaStream_t stream, bool upper)
{
    return launch_simple<double>(A, n, lda, strideA, batch, info, stream, upper);
}

int launch_cpotrf(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                  cudaStream_t stream, bool upper)
{
    if (n <= 64) return launch_cpotrf_warp(A, n, lda, strideA, batch, info, stream, upper);
    if (n <= 128) return launch_cpotrf_tiles(A, n, lda, strideA, batch, info, stream, upper);
    return launch_simple<float2>(reinterpret_cast<float2 *>(A), n, lda, strideA, batch, info,
                                 stream, upper);
}

int launch_zpotrf(double *A, int n, int lda, int64_t strideA, int batch, int *info,
                  cudaStream_t stream, bool upper)
{
    return launch_simple<double2>(reinterpret_cast<double2 *>(A), n, lda, strideA, batch, info,
                                  stream, upper);
}

}  // namespace bl
