// K1: batched SPOTRF for n <= 64, the matrix in the registers of one warp: for
// n <= 32 a group of N lanes per matrix (N = 32, 16 or 8, so one warp factors
// 1, 2 or 4 matrices); for 33 <= n <= 64 one warp per matrix, two rows a lane.
//
// Lane `row` of a group holds row `row` of its matrix, r[k] = a(row, k). The
// factorization is right-looking: at column j every lane publishes its current
// r[j] to a warp-private shared buffer, one __syncwarp, and every lane reads
// the pivot d_j and the column below it back as 16-byte broadcast loads. The
// pages measured this broadcast against shuffle chains and found the shuffles
// stalled on the MIO queue ("kernelbot-cholesky-930185", exp_s6 header, "THE
// SECOND FIX: n=32's SHUFFLES"); the buffer is double-buffered so no second
// sync is needed before the next column overwrites it.
//
// Per column, with s = rsqrt(d_j) and c_i = r[j] of lane i:
//   l_ij = c_i * s,  and for k > j:  r[k] -= (l_ij * s) * c_k      (= l_ij l_kj)
// so the broadcast column is read unscaled and no lane has to wait for another
// lane's scaling (one pre-scaled factor per lane instead of per entry).
//
// Rows and columns n .. N-1 of the register tile are an identity block, so the
// same unrolled code factors any n <= N. Lanes compute the whole row including
// the strict upper triangle of the register tile: values there are never read
// into a lower-triangle result and never stored.
#include <mutex>

#include "bl_common.cuh"

namespace bl {
namespace {

constexpr int kWarpsPerBlock = 1;  // one warp per block: blocks spread evenly over the SMs

template <int N, bool UP>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
potrf_warp_kernel(float *__restrict__ A, int n, int lda, int64_t strideA, int batch,
                  int *__restrict__ info)
{
    constexpr int G = 32 / N;  // matrices per warp
    __shared__ __align__(16) float colbuf[kWarpsPerBlock][2][32];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int grp = lane / N;
    const int row = lane - grp * N;
    const int64_t mat = ((int64_t)blockIdx.x * kWarpsPerBlock + warp) * G + grp;
    const bool valid = mat < batch;
    const bool live = valid && row < n;
    float *__restrict__ Ab = A + (valid ? mat * strideA : 0);
    pdl_wait();
    pdl_trigger();

    float r[N];
#pragma unroll
    for (int k = 0; k < N; ++k) {
        float v = (row == k) ? 1.0f : 0.0f;
        if (live && k <= row) v = Ab[lidx<UP>(row, k, lda)];
        r[k] = v;
    }

    float dm = 1.0f;  // this lane's pivot
#pragma unroll
    for (int j = 0; j < N; ++j) {
        if (j >= n) break;  // same n for every lane: uniform
        float *cb = colbuf[warp][j & 1];
        cb[lane] = r[j];
        __syncwarp();
        const float *col = cb + grp * N;
        const float d = col[j];
        const float s = rsqrt_approx(d);
        const float lij = r[j] * s;
        const float w = lij * s;
        r[j] = lij;
        dm = (row == j) ? d : dm;
        // columns j+1 .. N-1 of the broadcast column, read 4 at a time
#pragma unroll
        for (int q = (j + 1) / 4; q < N / 4; ++q) {
            const float4 c4 = reinterpret_cast<const float4 *>(col)[q];
            const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int k = 4 * q + t;
                if (k > j) r[k] = fmaf(-w, cv[t], r[k]);
            }
        }
    }

#pragma unroll
    for (int k = 0; k < N; ++k)
        if (live && k <= row) Ab[lidx<UP>(row, k, lda)] = r[k];
    // the diagonal from the lane's own pivot (sqrt(+Inf) = +Inf, like the
    // definition); info = the group's lowest row whose pivot failed
    if (live) Ab[lidx<UP>(row, row, lda)] = sqrt_approx(dm);
    const unsigned bad = __ballot_sync(0xffffffffu, live && !pivot_ok(dm));
    constexpr unsigned kGroupMask = (N == 32) ? 0xffffffffu : ((1u << (N & 31)) - 1u);
    const unsigned mine = (bad >> (grp * N)) & kGroupMask;
    if (valid && row == 0) info[mat] = mine ? __ffs(mine) : 0;
}

// n = 33 .. 64: one warp per matrix, lane i holds rows i (ra[k],
// k < 32) and i + 32 (rb[k], k < 64). Same column step as above; rows 0..31
// are finished after column 31, so from then on only rb is updated (a
// compile-time split, since the column loop is unrolled). The pivot test and
// the diagonal's square root are taken once at the end from each lane's own
// pivot (info by a warp ballot: the lowest failing row).
template <bool UP>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
potrf_warp64_kernel(float *__restrict__ A, int n, int lda, int64_t strideA, int batch,
                    int *__restrict__ info)
{
    __shared__ __align__(16) float colbuf[kWarpsPerBlock][2][64];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t mat = (int64_t)blockIdx.x * kWarpsPerBlock + warp;
    const bool valid = mat < batch;
    const int rowa = lane, rowb = lane + 32;
    const bool livea = valid && rowa < n, liveb = valid && rowb < n;
    float *__restrict__ Ab = A + (valid ? mat * strideA : 0);
    pdl_wait();
    pdl_trigger();

    float ra[32], rb[64];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        float v = (rowa == k) ? 1.0f : 0.0f;
        if (livea && k <= rowa) v = Ab[lidx<UP>(rowa, k, lda)];
        ra[k] = v;
    }
#pragma unroll
    for (int k = 0; k < 64; ++k) {
        float v = (rowb == k) ? 1.0f : 0.0f;
        if (liveb && k <= rowb) v = Ab[lidx<UP>(rowb, k, lda)];
        rb[k] = v;
    }

    float da = 1.0f, db = 1.0f;  // this lane's two pivots
#pragma unroll
    for (int j = 0; j < 64; ++j) {
        if (j >= n) break;
        float *cb = colbuf[warp][j & 1];
        if (j < 32) cb[lane] = ra[j];
        cb[lane + 32] = rb[j];
        __syncwarp();
        const float d = cb[j];
        const float s = rsqrt_approx(d);
        float wa = 0.0f;
        if (j < 32) {
            const float la = ra[j] * s;
            wa = la * s;
            ra[j] = la;
            da = (rowa == j) ? d : da;
        }
        const float lb = rb[j] * s;
        const float wb = lb * s;
        rb[j] = lb;
        db = (rowb == j) ? d : db;
#pragma unroll
        for (int q = (j + 1) / 4; q < 16; ++q) {
            const float4 c4 = reinterpret_cast<const float4 *>(cb)[q];
            const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int k = 4 * q + t;
                if (k > j) {
                    if (j < 32 && k < 32) ra[k] = fmaf(-wa, cv[t], ra[k]);
                    rb[k] = fmaf(-wb, cv[t], rb[k]);
                }
            }
        }
    }

#pragma unroll
    for (int k = 0; k < 32; ++k)
        if (livea && k <= rowa) Ab[lidx<UP>(rowa, k, lda)] = ra[k];
#pragma unroll
    for (int k = 0; k < 64; ++k)
        if (liveb && k <= rowb) Ab[lidx<UP>(rowb, k, lda)] = rb[k];
    // diagonal entries from the pivots (sqrt(+Inf) = +Inf, like the definition)
    if (livea) Ab[lidx<UP>(rowa, rowa, lda)] = sqrt_approx(da);
    if (liveb) Ab[lidx<UP>(rowb, rowb, lda)] = sqrt_approx(db);
    const unsigned fa = __ballot_sync(0xffffffffu, livea && !pivot_ok(da));
    const unsigned fb = __ballot_sync(0xffffffffu, liveb && !pivot_ok(db));
    if (valid && lane == 0) info[mat] = fa ? __ffs(fa) : (fb ? 32 + __ffs(fb) : 0);
}

// n = 33 .. 64 in two warps per matrix (small batches). Warp 0 holds rows i and i + 32 over
// columns 0..31 (ra, rb) and factors those columns exactly as the one-warp
// kernel does, publishing each column (rows 0..63) to a shared double buffer;
// warp 1 holds row i + 32 over columns 32..63 (rc), the trailing 32 x 32
// block, and applies every published column to it (the same scaled factor
// w = (c rsqrt d) rsqrt d as warp 0 takes for that row), then factors the block
// alone as the n <= 32 kernel does. One 64-thread barrier per column keeps the
// two in step; the serial path per lane drops from 2.5k to 1.5k FMAs.
template <bool UP>
__global__ void __maxnreg__(136)
potrf_warp64x2_kernel(float *__restrict__ A, int n, int lda, int64_t strideA, int batch,
                      int *__restrict__ info)
{
    __shared__ __align__(16) float col[2][64];  // column j, rows 0..63
    __shared__ __align__(16) float colb[2][32]; // warp 1's columns 32..63, rows 32..63
    __shared__ unsigned fail_a;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t mat = blockIdx.x;
    float *__restrict__ Ab = A + mat * strideA;
    pdl_wait();
    pdl_trigger();
    const int rowb = lane + 32;
    const bool liveb = rowb < n;

    if (warp == 0) {
        const int rowa = lane;  // < 32 < n
        float ra[32], rb[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            ra[k] = (k <= rowa) ? Ab[lidx<UP>(rowa, k, lda)] : 0.0f;
            rb[k] = liveb ? Ab[lidx<UP>(rowb, k, lda)] : 0.0f;
        }
        float da = 1.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            // n > 32 here, so this exit is never taken; it keeps the compiler
            // from hoisting work across columns (register pressure)
            if (j >= n) break;
            float *cb = col[j & 1];
            cb[lane] = ra[j];
            cb[lane + 32] = rb[j];
            named_bar_sync(1, 64);
            const float d = cb[j];
            const float s = rsqrt_approx(d);
            const float la = ra[j] * s, wa = la * s;
            const float lb = rb[j] * s, wb = lb * s;
            ra[j] = la;
            rb[j] = lb;
            da = (rowa == j) ? d : da;
#pragma unroll
            for (int q = (j + 1) / 4; q < 8; ++q) {
                const float4 c4 = reinterpret_cast<const float4 *>(cb)[q];
                const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int k = 4 * q + t;
                    if (k > j) {
                        ra[k] = fmaf(-wa, cv[t], ra[k]);
                        rb[k] = fmaf(-wb, cv[t], rb[k]);
                    }
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            if (k < rowa) Ab[lidx<UP>(rowa, k, lda)] = ra[k];
            if (liveb) Ab[lidx<UP>(rowb, k, lda)] = rb[k];
        }
        Ab[lidx<UP>(rowa, rowa, lda)] = sqrt_approx(da);
        const unsigned bad = __ballot_sync(0xffffffffu, !pivot_ok(da));
        if (lane == 0) fail_a = bad;
    } else {
        // rows 32..63 x columns 32..63; rows and columns n.. are the identity
        float rc[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            float v = (k == lane) ? 1.0f : 0.0f;
            if (liveb && k <= lane) v = Ab[lidx<UP>(rowb, (32 + k), lda)];
            rc[k] = v;
        }
#pragma unroll 1
        for (int j = 0; j < 32; ++j) {
            named_bar_sync(1, 64);
            const float *cb = col[j & 1];
            const float s = rsqrt_approx(cb[j]);
            const float w = (cb[lane + 32] * s) * s;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 c4 = reinterpret_cast<const float4 *>(cb + 32)[q];
                rc[4 * q] = fmaf(-w, c4.x, rc[4 * q]);
                rc[4 * q + 1] = fmaf(-w, c4.y, rc[4 * q + 1]);
                rc[4 * q + 2] = fmaf(-w, c4.z, rc[4 * q + 2]);
                rc[4 * q + 3] = fmaf(-w, c4.w, rc[4 * q + 3]);
            }
        }
        float db = 1.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (32 + j >= n) break;
            float *cb = colb[j & 1];
            cb[lane] = rc[j];
            __syncwarp();
            const float d = cb[j];
            const float s = rsqrt_approx(d);
            const float l = rc[j] * s, w = l * s;
            rc[j] = l;
            db = (lane == j) ? d : db;
#pragma unroll
            for (int q = (j + 1) / 4; q < 8; ++q) {
                const float4 c4 = reinterpret_cast<const float4 *>(cb)[q];
                const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int k = 4 * q + t;
                    if (k > j) rc[k] = fmaf(-w, cv[t], rc[k]);
                }
            }
        }
        if (liveb) {
#pragma unroll
            for (int k = 0; k < 32; ++k)
                if (k < lane) Ab[lidx<UP>(rowb, (32 + k), lda)] = rc[k];
            Ab[lidx<UP>(rowb, rowb, lda)] = sqrt_approx(db);
        }
        const unsigned bad = __ballot_sync(0xffffffffu, liveb && !pivot_ok(db));
        __syncwarp();
        named_bar_sync(2, 64);  // warp 0's failures are in fail_a
        if (lane == 0) {
            const unsigned fa = fail_a;
            info[mat] = fa ? __ffs(fa) : (bad ? 32 + __ffs(bad) : 0);
        }
        return;
    }
    named_bar_sync(2, 64);
}

template <int N, bool UP>
int launch_n(float *A, int n, int lda, int64_t strideA, int batch, int *info, cudaStream_t st)
{
    constexpr int G = 32 / N;
    const int64_t per_block = (int64_t)kWarpsPerBlock * G;
    const int64_t blocks = (batch + per_block - 1) / per_block;
    return launch_pdl(potrf_warp_kernel<N, UP>, dim3((unsigned)blocks), dim3(32 * kWarpsPerBlock), 0,
                      st, A, n, lda, strideA, batch, info);
}

// Blocks of the two-warp kernel that fit an SM (133 registers a thread: three
// warps per sub-partition).
constexpr int kX2BlocksPerSm = 6;

int sm_count()
{
    static std::once_flag once;
    static int sms = 0;
    std::call_once(once, [] {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            sms = 0;
    });
    return sms;
}

// n = 33 .. 64: two warps per matrix while the batch fits one wave of the
// two-warp kernel (lower latency: 6.4 against 7.7 us for one matrix, 7.5
// against 10.0 us for 152 on GB300); one warp per matrix above, where the
// two-warp kernel would need a second wave (1024 matrices: 11.3 against 17.3 us).
template <bool UP>
int launch_64(float *A, int n, int lda, int64_t strideA, int batch, int *info, cudaStream_t st)
{
    if ((int64_t)batch <= (int64_t)kX2BlocksPerSm * sm_count())
        return launch_pdl(potrf_warp64x2_kernel<UP>, dim3((unsigned)batch), dim3(64), 0, st, A,
                          n, lda, strideA, batch, info);
    const int64_t blocks = (batch + kWarpsPerBlock - 1) / kWarpsPerBlock;
    return launch_pdl(potrf_warp64_kernel<UP>, dim3((unsigned)blocks), dim3(32 * kWarpsPerBlock), 0,
                      st, A, n, lda, strideA, batch, info);
}

template <bool UP>
int launch_uplo(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                cudaStream_t stream)
{
    if (n <= 8) return launch_n<8, UP>(A, n, lda, strideA, batch, info, stream);
    if (n <= 16) return launch_n<16, UP>(A, n, lda, strideA, batch, info, stream);
    if (n <= 32) return launch_n<32, UP>(A, n, lda, strideA, batch, info, stream);
    return launch_64<UP>(A, n, lda, strideA, batch, info, stream);
}

}  // namespace

int launch_warp(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                cudaStream_t stream, bool upper)
{
    return upper ? launch_uplo<true>(A, n, lda, strideA, batch, info, stream)
                 : launch_uplo<false>(A, n, lda, strideA, batch, info, stream);
}

int attrs_warp(int n, cudaFuncAttributes *fa, int *threads, int *dyn_smem)
{
    cudaError_t e;
    if (n <= 8) e = cudaFuncGetAttributes(fa, potrf_warp_kernel<8, false>);
    else if (n <= 16) e = cudaFuncGetAttributes(fa, potrf_warp_kernel<16, false>);
    else if (n <= 32) e = cudaFuncGetAttributes(fa, potrf_warp_kernel<32, false>);
    else e = cudaFuncGetAttributes(fa, potrf_warp64_kernel<false>);  // the large-batch kernel
    *threads = 32 * kWarpsPerBlock;
    *dyn_smem = 0;
    return (int)e;
}

}  // namespace bl
