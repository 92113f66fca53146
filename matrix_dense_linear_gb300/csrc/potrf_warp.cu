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
#include "launch.cuh"

namespace bl {
namespace {

constexpr int kWarpsPerBlock = 1;  // one warp per block: blocks spread evenly over the SMs

// Row `row` of L, entries k0 .. k0+K-1: r[k] = l(row, k0 + k) where
// k0 + k <= row and `live`; other entries keep their values. Lower storage:
// 4-byte loads (the lanes of a warp read consecutive rows of one column).
// Upper storage: the row is contiguous in memory; 16-byte loads where `vec`
// and the whole quad lies on or left of the diagonal, 4-byte loads for the
// partial quad, so nothing right of the diagonal is read.
template <bool UP, int K>
__device__ __forceinline__ void load_row(float (&r)[K], const float *Ab, int row, int k0,
                                         int lda, bool live, bool vec)
{
    if constexpr (UP) {
        const float *p = Ab + (int64_t)row * lda + k0;
#pragma unroll
        for (int q = 0; q < K / 4; ++q) {
            if (live && vec && k0 + 4 * q + 3 <= row) {
                const float4 v = *reinterpret_cast<const float4 *>(p + 4 * q);
                r[4 * q] = v.x; r[4 * q + 1] = v.y; r[4 * q + 2] = v.z; r[4 * q + 3] = v.w;
            } else {
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    if (live && k0 + 4 * q + t <= row) r[4 * q + t] = p[4 * q + t];
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < K; ++k)
            if (live && k0 + k <= row) r[k] = Ab[lidx<false>(row, k0 + k, lda)];
    }
}

// The inverse of load_row: entries k0 + k <= row of the row go back to memory.
template <bool UP, int K>
__device__ __forceinline__ void store_row(const float (&r)[K], float *Ab, int row, int k0,
                                          int lda, bool live, bool vec)
{
    if constexpr (UP) {
        float *p = Ab + (int64_t)row * lda + k0;
#pragma unroll
        for (int q = 0; q < K / 4; ++q) {
            if (live && vec && k0 + 4 * q + 3 <= row) {
                *reinterpret_cast<float4 *>(p + 4 * q) =
                    make_float4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
            } else {
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    if (live && k0 + 4 * q + t <= row) p[4 * q + t] = r[4 * q + t];
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < K; ++k)
            if (live && k0 + k <= row) Ab[lidx<false>(row, k0 + k, lda)] = r[k];
    }
}

// 16-byte loads of the upper storage need A, lda and strideA in multiples of 4 floats
__device__ __forceinline__ bool vec_ok(const float *A, int lda, int64_t strideA)
{
    return ((reinterpret_cast<uintptr_t>(A) & 15) == 0) && ((lda & 3) == 0) &&
           ((strideA & 3) == 0);
}

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

    const bool vec = UP && vec_ok(A, lda, strideA);
    float r[N];
#pragma unroll
    for (int k = 0; k < N; ++k) r[k] = (row == k) ? 1.0f : 0.0f;
    load_row<UP>(r, Ab, row, 0, lda, live, vec);

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
        // by pairs of columns with the paired single-precision FMA (two
        // fused multiply-adds, each rounded as fmaf, in one instruction); a
        // single column where the pair straddles j
        const float2 nw = make_float2(-w, -w);
#pragma unroll
        for (int q = (j + 1) / 4; q < N / 4; ++q) {
            const float4 c4 = reinterpret_cast<const float4 *>(col)[q];
            const float2 cp[2] = {make_float2(c4.x, c4.y), make_float2(c4.z, c4.w)};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int k = 4 * q + 2 * h;
                if (k > j) {
                    const float2 t = __ffma2_rn(nw, cp[h], make_float2(r[k], r[k + 1]));
                    r[k] = t.x; r[k + 1] = t.y;
                } else if (k + 1 > j) {
                    r[k + 1] = fmaf(-w, cp[h].y, r[k + 1]);
                }
            }
        }
    }

    asm volatile("" : "+r"(lda));  // no load address lives to the stores
    store_row<UP>(r, Ab, row, 0, lda, live, vec);
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
    // No early trigger here: the next launch's warps would take the free slots
    // of this one's SMs (up to three warps per sub-partition at 153 registers)
    // and then start unevenly (1024 matrices: 14.4 against 11.9 us a call in a
    // chain of launches); the implicit trigger at exit keeps them out.
    pdl_wait();

    const bool vec = UP && vec_ok(A, lda, strideA);
    float ra[32], rb[64];
#pragma unroll
    for (int k = 0; k < 32; ++k) ra[k] = (rowa == k) ? 1.0f : 0.0f;
#pragma unroll
    for (int k = 0; k < 64; ++k) rb[k] = (rowb == k) ? 1.0f : 0.0f;
    load_row<UP>(ra, Ab, rowa, 0, lda, livea, vec);
    load_row<UP>(rb, Ab, rowb, 0, lda, liveb, vec);

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

    // lda made opaque before the stores: otherwise the compiler keeps the load
    // addresses alive across the whole factorization to reuse them here
    // (n = 64: 211 against 153 registers a thread; two warps: 133 against 114)
    asm volatile("" : "+r"(lda));
    store_row<UP>(ra, Ab, rowa, 0, lda, livea, vec);
    store_row<UP>(rb, Ab, rowb, 0, lda, liveb, vec);
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
__global__ void __launch_bounds__(64, 8)
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
    const bool vec = UP && vec_ok(A, lda, strideA);

    if (warp == 0) {
        const int rowa = lane;  // < 32 < n
        float ra[32], rb[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) ra[k] = rb[k] = 0.0f;
        load_row<UP>(ra, Ab, rowa, 0, lda, true, vec);
        load_row<UP>(rb, Ab, rowb, 0, lda, liveb, vec);
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
        asm volatile("" : "+r"(lda));  // no load address lives to the stores
        store_row<UP>(ra, Ab, rowa, 0, lda, true, vec);  // its diagonal is rewritten below
        store_row<UP>(rb, Ab, rowb, 0, lda, liveb, vec);
        Ab[lidx<UP>(rowa, rowa, lda)] = sqrt_approx(da);
        const unsigned bad = __ballot_sync(0xffffffffu, !pivot_ok(da));
        if (lane == 0) fail_a = bad;
    } else {
        // rows 32..63 x columns 32..63; rows and columns n.. are the identity
        float rc[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) rc[k] = (k == lane) ? 1.0f : 0.0f;
        load_row<UP>(rc, Ab, rowb, 32, lda, liveb, vec);
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
        asm volatile("" : "+r"(lda));  // no load address lives to the stores
        store_row<UP>(rc, Ab, rowb, 32, lda, liveb, vec);  // its diagonal is rewritten below
        if (liveb) Ab[lidx<UP>(rowb, rowb, lda)] = sqrt_approx(db);
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

template <int N, bool UP>
int launch_n(float *A, int n, int lda, int64_t strideA, int batch, int *info, cudaStream_t st)
{
    constexpr int G = 32 / N;
    const int64_t per_block = (int64_t)kWarpsPerBlock * G;
    const int64_t blocks = (batch + per_block - 1) / per_block;
    return launch_pdl(potrf_warp_kernel<N, UP>, dim3((unsigned)blocks),
                      dim3(32 * kWarpsPerBlock), 0,
                      st, A, n, lda, strideA, batch, info);
}

// The two-warp kernel runs while its blocks put at most two warps on an SM
// sub-partition (four blocks per SM); above, one warp per matrix is faster
// (760 matrices of order 64: 10.3 against 12.6 us).
constexpr int kX2BlocksPerSm = 4;

// n = 33 .. 64: two warps per matrix for small batches (lower latency: one
// matrix 6.4 against 7.7 us, 608 matrices 8.9 against 10.1 us on GB300), one
// warp per matrix above.
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
