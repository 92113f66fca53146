// CPOTRF for n <= 64 in registers: the complex Hermitian form of K1's
// lane-per-row factorization (A = L L^H, lower). The upper storage keeps
// U = L^H, and conj(A) = A^T is Hermitian with the lower factor conj(L) = U^T:
// so in that storage a lane reads row i of A^T (column i of the stored upper
// triangle, as is), factors conj(A) by the same steps and writes conj(L) back
// in place, which is U. No conjugation anywhere (and, negation being exact,
// the same bits as conjugating on the way in and out).
//
// n <= 32: a group of N lanes (N = 32, 16 or 8) factors one matrix, so one
// warp factors 1, 2 or 4. n = 33 .. 64: two warps a matrix, warp 0 holding
// rows 0..31 (columns 0..31 only: its rows end there) and warp 1 rows 32..63;
// a 64-thread barrier a column while both publish (columns 0..31), then warp 1
// goes on alone with __syncwarp. Lane `row` holds row `row`, r[k] = a(row, k).
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

template <bool UP>
__global__ void __launch_bounds__(64)
cpotrf_warp64_kernel(float2 *__restrict__ A, int n, int lda, int64_t strideA, int batch,
                     int *__restrict__ info)
{
    __shared__ __align__(16) float2 colbuf[2][64];
    __shared__ unsigned fail0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t mat = blockIdx.x;  // the grid is the batch
    float2 *__restrict__ Ab = A + mat * strideA;
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        const int row = lane;  // < 32 < n
        float2 r[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) r[k] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (k <= row) r[k] = Ab[lidx<UP>(row, k, lda)];
        float dm = 1.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            // n > 32 here, so this exit is never taken; it keeps the compiler
            // from hoisting work across columns (register pressure)
            if (j >= n) break;
            float2 *cb = colbuf[j & 1];
            cb[row] = r[j];
            named_bar_sync(1, 64);
            const float d = column_step(r, cb, j);
            dm = (row == j) ? d : dm;
        }
        asm volatile("" : "+r"(lda));  // no load address lives to the stores
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (k < row) Ab[lidx<UP>(row, k, lda)] = r[k];
        Ab[lidx<UP>(row, row, lda)] = make_float2(sqrt_approx(dm), 0.0f);
        const unsigned bad = __ballot_sync(0xffffffffu, !pivot_ok(dm));
        if (lane == 0) fail0 = bad;
    } else {
        const int row = 32 + lane;
        const bool live = row < n;
        float2 r[64];  // rows and columns n.. are the identity
#pragma unroll
        for (int k = 0; k < 64; ++k) r[k] = make_float2(row == k ? 1.0f : 0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < 64; ++k)
            if (live && k <= row) r[k] = Ab[lidx<UP>(row, k, lda)];
        float dm = 1.0f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
            if (j >= n) break;  // uniform
            float2 *cb = colbuf[j & 1];
            cb[row] = r[j];
            // columns 32.. live in this warp's rows only; warp 0 never reads
            // an entry that this warp writes after the last joint barrier
            if (j < 32) named_bar_sync(1, 64);
            else __syncwarp();
            const float d = column_step(r, cb, j);
            dm = (row == j) ? d : dm;
        }
        asm volatile("" : "+r"(lda));
#pragma unroll
        for (int k = 0; k < 64; ++k)
            if (live && k < row) Ab[lidx<UP>(row, k, lda)] = r[k];
        if (live) Ab[lidx<UP>(row, row, lda)] = make_float2(sqrt_approx(dm), 0.0f);
        const unsigned bad = __ballot_sync(0xffffffffu, live && !pivot_ok(dm));
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
