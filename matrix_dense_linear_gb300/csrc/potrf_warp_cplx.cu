// CPOTRF for n <= 64 in registers: the complex Hermitian form of K1's
// lane-per-row factorization (A = L L^H, lower). The upper storage keeps
// U = L^H, and conj(A) = A^T is Hermitian with the lower factor conj(L) = U^T:
// so in that storage a lane reads row i of A^T (column i of the stored upper
// triangle, as is), factors conj(A) by the same steps and writes conj(L) back
// in place, which is U. No conjugation anywhere (and, negation being exact,
// the same bits as conjugating on the way in and out).
//
// n <= 32: a group of N lanes (N = 32, 16 or 8) factors one matrix, so one
// warp factors 1, 2 or 4; lane `row` holds row `row`, r[k] = a(row, k).
// n = 33 .. 64: two warps a matrix, split by columns: warp 0 holds rows i and
// i + 32 over columns 0..31 and factors those columns (a 64-thread barrier a
// column); warp 1 holds row i + 32 over columns 32..63, applies each published
// column to that whole trailing block (uniform work, a rolled loop), then
// factors the block alone. This keeps the unrolled code near 6k instructions a
// matrix: holding whole rows instead (warp 0 rows 0..31, warp 1 rows 32..63,
// ~10k instructions) ran 1024 matrices of order 64 in 72 against 40 us.
// Column step j, with c_i = r[j] of lane i published unscaled to a
// warp-private, double-buffered shared column and s = rsqrt(re(d_j)):
//   l_ij = c_i s,   and for k > j:  r[k] -= (l_ij s) conj(c_k)   (= l_ij conj(l_kj))
// The pivot is the real part of the diagonal: its imaginary part is never
// read, and the diagonal is written as sqrt(d) + 0i from each lane's own pivot
// at the end (info = the group's lowest row whose pivot failed, as in the
// real kernel). Rows and columns n .. N-1 are an identity block; entries right
// of the diagonal in the register tile are computed but never stored.
#include <mutex>

#include "bl_common.cuh"
#include "launch.cuh"

namespace bl {
namespace {

// One column step of a lane's row r[0..K-1]: the column's entries sit
// unscaled in col[0..], d = re(col[j]) its pivot. Returns d.
template <int K>
__device__ __forceinline__ float column_step(float2 (&r)[K], const float2 *col, int j)
{
    const float d = col[j].x;
    const float s = rsqrt_approx(d);
    const float2 l = make_float2(r[j].x * s, r[j].y * s);
    const float2 w = make_float2(l.x * s, l.y * s);
    r[j] = l;
#pragma unroll
    for (int q = (j + 1) / 2; q < K / 2; ++q) {
        const float4 c2 = reinterpret_cast<const float4 *>(col)[q];
        const float2 cv[2] = {make_float2(c2.x, c2.y), make_float2(c2.z, c2.w)};
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int k = 2 * q + t;
            if (k > j) {  // r[k] -= w conj(c_k)
                r[k].x = fmaf(-w.x, cv[t].x, fmaf(-w.y, cv[t].y, r[k].x));
                r[k].y = fmaf(-w.y, cv[t].x, fmaf(w.x, cv[t].y, r[k].y));
            }
        }
    }
    return d;
}

template <int N, bool UP>
__global__ void __launch_bounds__(32)
cpotrf_warp_kernel(float2 *__restrict__ A, int n, int lda, int64_t strideA, int batch,
                   int *__restrict__ info)
{
    constexpr int G = 32 / N;  // matrices per warp
    __shared__ __align__(16) float2 colbuf[2][32];

    const int lane = threadIdx.x & 31;
    const int grp = lane / N;
    const int row = lane - grp * N;
    const int64_t mat = (int64_t)blockIdx.x * G + grp;
    const bool valid = mat < batch;
    const bool live = valid && row < n;
    float2 *__restrict__ Ab = A + (valid ? mat * strideA : 0);
    pdl_wait();
    pdl_trigger();

    float2 r[N];
#pragma unroll
    for (int k = 0; k < N; ++k) r[k] = make_float2(row == k ? 1.0f : 0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < N; ++k)
        if (live && k <= row) r[k] = Ab[lidx<UP>(row, k, lda)];

    float dm = 1.0f;  // this lane's pivot
#pragma unroll
    for (int j = 0; j < N; ++j) {
        if (j >= n) break;  // same n for every lane: uniform
        float2 *cb = colbuf[j & 1];
        cb[lane] = r[j];
        __syncwarp();
        const float d = column_step(r, cb + grp * N, j);
        dm = (row == j) ? d : dm;
    }

    asm volatile("" : "+r"(lda));  // no load address lives to the stores
#pragma unroll
    for (int k = 0; k < N; ++k)
        if (live && k < row) Ab[lidx<UP>(row, k, lda)] = r[k];
    if (live) Ab[lidx<UP>(row, row, lda)] = make_float2(sqrt_approx(dm), 0.0f);
    const unsigned bad = __ballot_sync(0xffffffffu, live && !pivot_ok(dm));
    constexpr unsigned kGroupMask = (N == 32) ? 0xffffffffu : ((1u << (N & 31)) - 1u);
    const unsigned mine = (bad >> (grp * N)) & kGroupMask;
    if (valid && row == 0) info[mat] = mine ? __ffs(mine) : 0;
}

// six blocks an SM (167 registers a thread; 204 when left to the compiler)
template <bool UP>
__global__ void __launch_bounds__(64, 6)
cpotrf_warp64_kernel(float2 *__restrict__ A, int n, int lda, int64_t strideA, int batch,
                     int *__restrict__ info)
{
    __shared__ __align__(16) float2 col[2][64];   // column j < 32, rows 0..63
    __shared__ __align__(16) float2 colb[2][32];  // warp 1's columns 32.., rows 32..63
    __shared__ unsigned fail0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t mat = blockIdx.x;  // the grid is the batch
    float2 *__restrict__ Ab = A + mat * strideA;
    pdl_wait();
    pdl_trigger();
    const int rowb = 32 + lane;
    const bool liveb = rowb < n;

    if (warp == 0) {
        // rows lane and lane + 32 over columns 0..31; both updates read the
        // same broadcast entries (rows 0..31 of the column)
        const int rowa = lane;  // < 32 < n
        float2 ra[32], rb[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) ra[k] = rb[k] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (k <= rowa) ra[k] = Ab[lidx<UP>(rowa, k, lda)];
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (liveb) rb[k] = Ab[lidx<UP>(rowb, k, lda)];
        float da = 1.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            // n > 32 here, so this exit is never taken; it keeps the compiler
            // from hoisting work across columns (register pressure)
            if (j >= n) break;
            float2 *cb = col[j & 1];
            cb[rowa] = ra[j];
            cb[rowb] = rb[j];
            named_bar_sync(1, 64);
            const float d = cb[j].x;
            const float s = rsqrt_approx(d);
            const float2 la = make_float2(ra[j].x * s, ra[j].y * s);
            const float2 lb = make_float2(rb[j].x * s, rb[j].y * s);
            const float2 wa = make_float2(la.x * s, la.y * s);
            const float2 wb = make_float2(lb.x * s, lb.y * s);
            ra[j] = la;
            rb[j] = lb;
            da = (rowa == j) ? d : da;
#pragma unroll
            for (int q = (j + 1) / 2; q < 16; ++q) {
                const float4 c2 = reinterpret_cast<const float4 *>(cb)[q];
                const float2 cv[2] = {make_float2(c2.x, c2.y), make_float2(c2.z, c2.w)};
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int k = 2 * q + t;
                    if (k > j) {
                        ra[k].x = fmaf(-wa.x, cv[t].x, fmaf(-wa.y, cv[t].y, ra[k].x));
                        ra[k].y = fmaf(-wa.y, cv[t].x, fmaf(wa.x, cv[t].y, ra[k].y));
                        rb[k].x = fmaf(-wb.x, cv[t].x, fmaf(-wb.y, cv[t].y, rb[k].x));
                        rb[k].y = fmaf(-wb.y, cv[t].x, fmaf(wb.x, cv[t].y, rb[k].y));
                    }
                }
            }
        }
        asm volatile("" : "+r"(lda));  // no load address lives to the stores
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (k < rowa) Ab[lidx<UP>(rowa, k, lda)] = ra[k];
        Ab[lidx<UP>(rowa, rowa, lda)] = make_float2(sqrt_approx(da), 0.0f);
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (liveb) Ab[lidx<UP>(rowb, k, lda)] = rb[k];
        const unsigned bad = __ballot_sync(0xffffffffu, !pivot_ok(da));
        if (lane == 0) fail0 = bad;
    } else {
        // row lane + 32 over columns 32..63, the trailing block; rows and
        // columns n.. are the identity
        float2 rc[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) rc[k] = make_float2(k == lane ? 1.0f : 0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (liveb && k <= lane) rc[k] = Ab[lidx<UP>(rowb, 32 + k, lda)];
        // columns 0..31 as warp 0 publishes them: the same factor w that warp 0
        // takes for this row, every entry of the block (a loop, not unrolled)
#pragma unroll 1
        for (int j = 0; j < 32; ++j) {
            named_bar_sync(1, 64);
            const float2 *cb = col[j & 1];
            const float s = rsqrt_approx(cb[j].x);
            const float2 c = cb[rowb];
            const float2 l = make_float2(c.x * s, c.y * s);
            const float2 w = make_float2(l.x * s, l.y * s);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float4 c2 = reinterpret_cast<const float4 *>(cb + 32)[q];
                const float2 cv[2] = {make_float2(c2.x, c2.y), make_float2(c2.z, c2.w)};
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    float2 &e = rc[2 * q + t];
                    e.x = fmaf(-w.x, cv[t].x, fmaf(-w.y, cv[t].y, e.x));
                    e.y = fmaf(-w.y, cv[t].x, fmaf(w.x, cv[t].y, e.y));
                }
            }
        }
        // then the block alone, as the n <= 32 kernel factors a matrix
        float dc = 1.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (32 + j >= n) break;  // uniform
            float2 *cb = colb[j & 1];
            cb[lane] = rc[j];
            __syncwarp();
            const float d = column_step(rc, cb, j);
            dc = (lane == j) ? d : dc;
        }
        asm volatile("" : "+r"(lda));
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (liveb && k < lane) Ab[lidx<UP>(rowb, 32 + k, lda)] = rc[k];
        if (liveb) Ab[lidx<UP>(rowb, rowb, lda)] = make_float2(sqrt_approx(dc), 0.0f);
        const unsigned bad = __ballot_sync(0xffffffffu, liveb && !pivot_ok(dc));
        named_bar_sync(2, 64);
        if (lane == 0) info[mat] = fail0 ? __ffs(fail0) : (bad ? 32 + __ffs(bad) : 0);
        return;
    }
    named_bar_sync(2, 64);
}

template <int N, bool UP>
int launch_n(float2 *A, int n, int lda, int64_t strideA, int batch, int *info, cudaStream_t st)
{
    constexpr int G = 32 / N;
    const unsigned blocks = (unsigned)((batch + G - 1) / G);
    return launch_pdl(cpotrf_warp_kernel<N, UP>, dim3(blocks), dim3(32), 0, st, A, n, lda,
                      strideA, batch, info);
}

template <bool UP>
int launch_u(float2 *A, int n, int lda, int64_t strideA, int batch, int *info, cudaStream_t st)
{
    if (n > 32)
        return launch_pdl(cpotrf_warp64_kernel<UP>, dim3((unsigned)batch), dim3(64), 0, st, A, n,
                          lda, strideA, batch, info);
    if (n <= 8) return launch_n<8, UP>(A, n, lda, strideA, batch, info, st);
    if (n <= 16) return launch_n<16, UP>(A, n, lda, strideA, batch, info, st);
    return launch_n<32, UP>(A, n, lda, strideA, batch, info, st);
}

}  // namespace

int launch_cpotrf_warp(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                       cudaStream_t stream, bool upper)
{
    if (n < 1 || n > 64) return -1;
    float2 *Ac = reinterpret_cast<float2 *>(A);
    return upper ? launch_u<true>(Ac, n, lda, strideA, batch, info, stream)
                 : launch_u<false>(Ac, n, lda, strideA, batch, info, stream);
}

}  // namespace bl
