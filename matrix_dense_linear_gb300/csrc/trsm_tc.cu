// Panel solve of the blocked path with the tensor cores doing the block updates:
//     L21 = A21 L11^{-T}      (A21: the rows below the 128 x 128 diagonal block)
// as a blocked forward substitution over four 32-column blocks j:
//     X_j = (A_j - sum_{i<j} X_i L_ji^T) L_jj^{-T}.
// One block of 128 threads takes 128 rows. Tensor memory holds -(A21 rows)
// (lane = row, column = panel column). For j = 0..3 every thread reads its
// row's 32 columns of block j back, solves them against the 32 x 32 diagonal
// block L_jj with the reciprocal-root scaling of K2 (one row per thread, the
// trsm_panel kernel of "kernelbot-cholesky-930185"), stores the finished X_j
// and stages it (3xTF32 split, K-major) as the A operand of one group of
// tcgen05.mma that adds X_j L_{k,j}^T to every later column block k > j in
// tensor memory. Three quarters of the flops run on the tensor cores; only the
// 32-column triangular solves stay on the FP32 pipes.
//
// The off-diagonal rows of L11 are staged one column block at a time (fetched
// into registers while the previous block is solved), which keeps the block's
// shared memory at 75 KB: three blocks share an SM. Needs 16-byte aligned
// panels (the caller falls back to the FP32 kernel otherwise). Every wait is
// bounded; a block that gives up marks info = -1. The upper storage (uplo =
// 'U') changes only the addresses: a row of L is contiguous there.
#include <mutex>

#include "bl_common.cuh"
#include "launch.cuh"
#include "tc_sm100.cuh"

namespace bl {
namespace {

constexpr uint32_t kLbo = 128;
constexpr uint32_t kSbo = 8 * 128 + 16;          // K = 32 per row group, +16 B (banks)
constexpr uint32_t kXTile = 16 * kSbo;           // 128 rows
constexpr long long kWaitCycles = 2000000000LL;

// rows of L_{k,j}, k > j, for column block j
__host__ __device__ constexpr uint32_t lt_rows(int j) { return (uint32_t)(96 - 32 * j); }

// Shared memory: the X operand (hi, lo); the off-diagonal rows of one column
// block of L11 at a time (hi, lo; sized for block 0); the four diagonal
// blocks; the reciprocal diagonal. 75 KB: three blocks share an SM.
constexpr uint32_t kOffX = 0;
constexpr uint32_t kOffLt = 2 * kXTile;
constexpr uint32_t kLtBytes = 2 * (lt_rows(0) / 8) * kSbo;
constexpr uint32_t kOffLd = kOffLt + kLtBytes;
constexpr uint32_t kOffRinv = kOffLd + 4 * 32 * 32 * 4;
constexpr int kSmemBytes = (int)(kOffRinv + 128 * 4);

// failure injection for the give-up test (see set_fail_first_wait in launch.cuh)
__device__ int g_fail_first_wait;

__device__ __forceinline__ uint32_t core_off(int r, int q)
{
    return (uint32_t)(r >> 3) * kSbo + (uint32_t)q * kLbo + (uint32_t)(r & 7) * 16;
}

// Column block j of L11 below its diagonal block, L_{k,j} for k > j, in 4 x 4
// pieces (rows i..i+3 of columns 4q..4q+3 of the block), row quads fastest.
// A thread owns pieces tid and tid + 128: load() fetches them into registers
// as four 16-byte loads (down the columns in the lower storage, along the rows
// in the upper one), stage() splits them into the K-major hi/lo operand tiles.
template <bool UP>
struct LtPieces {
    float4 v[2][4];  // lower storage: [column][4 rows]; upper: [row][4 columns]
    __device__ __forceinline__ void load(const float *L11, int lda, int j, int tid)
    {
        const int nrq = (int)lt_rows(j) / 4;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int b = tid + 128 * u;
            if (b < nrq * 8) {
                const int rq = b % nrq, q = b / nrq;
                const float *src = L11 + lidx<UP>(32 * (j + 1) + 4 * rq, 32 * j + 4 * q, lda);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    v[u][c] = *reinterpret_cast<const float4 *>(src + (int64_t)c * lda);
            }
        }
    }
    __device__ __forceinline__ void stage(uint8_t *hi, int j, int tid) const
    {
        const int nrq = (int)lt_rows(j) / 4;
        uint8_t *lo = hi + lt_rows(j) / 8 * kSbo;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int b = tid + 128 * u;
            if (b < nrq * 8) {
                const int rq = b % nrq, q = b / nrq;
                const float cv[4][4] = {{v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w},
                                        {v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w},
                                        {v[u][2].x, v[u][2].y, v[u][2].z, v[u][2].w},
                                        {v[u][3].x, v[u][3].y, v[u][3].z, v[u][3].w}};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float h[4], l[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        tc::split_tf32(UP ? cv[i][c] : cv[c][i], h[c], l[c]);
                    const uint32_t off = core_off(4 * rq + i, q);
                    *reinterpret_cast<float4 *>(hi + off) = make_float4(h[0], h[1], h[2], h[3]);
                    *reinterpret_cast<float4 *>(lo + off) = make_float4(l[0], l[1], l[2], l[3]);
                }
            }
        }
    }
};

// FUSED (the panel's rows are the whole trailing matrix, m <= 128): the
// trailing update A22 -= L21 L21^T is done here too, as one more MMA group per
// column block, D += X_j X_j^T in a second 128-column accumulator, subtracted
// from A22's lower triangle at the end (no separate update launch; L21 is not
// read back).
template <bool UP, bool FUSED>
__global__ void __launch_bounds__(128, FUSED ? 2 : 3)
trsm_tc_kernel(float *__restrict__ A, int n, int lda, int64_t strideA, int c0, int nrb,
               int *__restrict__ info)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint32_t tmem_base;
    __shared__ __align__(8) uint64_t mbar;
    __shared__ int sh_err;

    // one-dimensional grid, the row block fastest: a matrix's row blocks run
    // together and share its L11 through L2
    const int64_t mat = blockIdx.x / nrb;
    const int rb = (int)(blockIdx.x % nrb);
    // launched as a programmatic dependent: wait for the previous kernel's
    // writes, then let the next kernel of the stream start launching
    pdl_wait();
    pdl_trigger();
    if (block_skip(info, mat)) return;
    float *__restrict__ Ab = A + mat * strideA;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int R = c0 + 128 + rb * 128 + tid;  // this thread's row
    const bool live = R < n;
    const int64_t xs = UP ? 1 : lda;  // step between the columns of one row
    const float *L11 = Ab + c0 + (int64_t)c0 * lda;         // L11(i, k) = L11[lidx(i, k)]
    float *Ld = reinterpret_cast<float *>(smem + kOffLd);    // Ld[j*1024 + t*32 + k] = L(32j+k, 32j+t)
    float *rinv = reinterpret_cast<float *>(smem + kOffRinv);
    uint8_t *Lt = smem + kOffLt;

    if (tid == 0) {
        sh_err = 0;
        tc::mbar_init(&mbar, 1);
        tc::fence_mbar_init();
    }
    constexpr uint32_t kCols = FUSED ? 256 : 128;
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, kCols);
        tc::tmem_relinquish();
    }

    // diagonal blocks of L11 (lower part) by asynchronous copies
    for (int col = warp; col < 128; col += 4) {
        const int j = col >> 5, t = col & 31;
        for (int k = t + lane; k < 32; k += 32)
            cp_async4(Ld + j * 1024 + t * 32 + k, L11 + lidx<UP>(32 * j + k, col, lda));
    }
    cp_async_commit();

    // -A21 rows, this thread's row: column chunks of 32 (one column at a time in
    // the lower storage). In the upper storage a row is contiguous: the warp
    // reads its 32 rows four at a time, a quarter warp a row's 128 bytes, and
    // passes them through its slice of the X region (free until the first
    // X operand is staged), so that every load is a whole line
    const float *g = Ab + (live ? lidx<UP>(R, c0, lda) : 0);  // g[c * xs] = (R, c0 + c)
    const int Rw = c0 + 128 + rb * 128 + 32 * warp;            // the warp's first row
    float *tb = reinterpret_cast<float *>(smem + kOffX) + warp * (32 * 36);  // [32][36]
    auto load_chunk = [&](int q, float (&v)[32]) {
        if constexpr (UP) {
            __syncwarp();  // the slice's previous contents are read
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = 4 * i + (lane >> 3), cq = lane & 7;
                const float4 a = Rw + r < n
                    ? *reinterpret_cast<const float4 *>(Ab + (c0 + 32 * q + 4 * cq) +
                                                        (int64_t)(Rw + r) * lda)
                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                *reinterpret_cast<float4 *>(tb + r * 36 + 4 * cq) = a;
            }
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
                const float4 a = *reinterpret_cast<const float4 *>(tb + lane * 36 + c);
                v[c] = -a.x; v[c + 1] = -a.y; v[c + 2] = -a.z; v[c + 3] = -a.w;
            }
        } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = live ? -g[(int64_t)(32 * q + c) * xs] : 0.0f;
        }
    };
    // the off-diagonal rows of L11's column block 0 and the first half of the
    // row travel together (one memory round trip instead of two); the second
    // half follows once the first is in tensor memory
    LtPieces<UP> pc;
    pc.load(L11, lda, 0, tid);
    float v0[32], v1[32];
    load_chunk(0, v0);
    load_chunk(1, v1);
    pc.stage(Lt, 0, tid);

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base;
    const uint32_t tlane = tmem + ((uint32_t)(32 * warp) << 16);
    tc::tmem_st32(tlane, v0);
    tc::tmem_st32(tlane + 32, v1);
    load_chunk(2, v0);
    load_chunk(3, v1);
    tc::tmem_st32(tlane + 64, v0);
    tc::tmem_st32(tlane + 96, v1);
    cp_async_wait<0>();
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    rinv[tid] = 1.0f / Ld[(tid >> 5) * 1024 + (tid & 31) * 33];
    __syncthreads();

    const uint32_t sbase = tc::smem_u32(smem);
    // the MMA group committed last and not yet seen complete (thread 0; -1: none):
    // a block that gives up waits for it before releasing tensor memory
    int pend = -1;
#pragma unroll 1
    for (int j = 0; j < 4; ++j) {
        if (j > 0) {
            if (tid == 0) {
                if (!(j == 1 && injected_failure(g_fail_first_wait, mat)) &&
                    tc::mbar_wait(&mbar, (j - 1) & 1, kWaitCycles))
                    pend = -1;
                else sh_err = 1;
            }
            tc::fence_before_sync();
            __syncthreads();
            if (sh_err) break;
            tc::fence_after_sync();
            // the operand tiles are free again: the off-diagonal rows of block j
            if (j < 3) pc.stage(Lt, j, tid);
        }
        // block j+1's off-diagonal rows travel while block j is solved
        if (j + 1 < 3) pc.load(L11, lda, j + 1, tid);
        float x[32];
        tc::tmem_ld32(tlane + 32 * j, x);
        const float *Lj = Ld + j * 1024;
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            x[t] = -x[t] * rinv[32 * j + t];
            const float *Lt_ = Lj + t * 32;
#pragma unroll
            for (int q = (t + 1) / 4; q < 8; ++q) {
                const float4 l4 = reinterpret_cast<const float4 *>(Lt_)[q];
                const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int k = 4 * q + u;
                    if (k > t) x[k] = fmaf(x[t], lv[u], x[k]);  // x[k] holds -(...)
                }
            }
        }
        if constexpr (UP) {
            // through the warp's slice of the X region (the MMAs of block j - 1
            // that read it are complete), a quarter warp writing a row's 128 bytes
#pragma unroll
            for (int t = 0; t < 32; t += 4)
                *reinterpret_cast<float4 *>(tb + lane * 36 + t) =
                    make_float4(x[t], x[t + 1], x[t + 2], x[t + 3]);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = 4 * i + (lane >> 3), cq = lane & 7;
                if (Rw + r < n)
                    *reinterpret_cast<float4 *>(Ab + (c0 + 32 * j + 4 * cq) + (int64_t)(Rw + r) * lda) =
                        *reinterpret_cast<const float4 *>(tb + r * 36 + 4 * cq);
            }
            __syncthreads();  // every warp is done with its slice before X is staged
        } else if (live) {
            float *out = Ab + lidx<UP>(R, c0 + 32 * j, lda);
#pragma unroll
            for (int t = 0; t < 32; ++t) out[(int64_t)t * xs] = x[t];
        }
        if (j == 3 && !FUSED) break;
        // X_j as the A operand (K-major, hi/lo)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float h[4], l[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) tc::split_tf32(x[4 * q + u], h[u], l[u]);
            const uint32_t off = core_off(tid, q);
            *reinterpret_cast<float4 *>(smem + kOffX + off) = make_float4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<float4 *>(smem + kOffX + kXTile + off) =
                make_float4(l[0], l[1], l[2], l[3]);
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (tid == 0 && j < 3) {
            // -A[:, 32(j+1):] += X_j L_{k,j}^T   (M = 128, N = 96 - 32j, K = 32)
            const uint32_t N = lt_rows(j);
            const uint32_t idesc = tc::idesc_tf32(128, N);
            const uint32_t xh = sbase + kOffX, xl = xh + kXTile;
            const uint32_t bh = sbase + kOffLt, bl = bh + N / 8 * kSbo;
            const uint32_t d = tmem + 32 * (j + 1);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint32_t ko = ks * 2 * kLbo;
                tc::mma_tf32(d, tc::smem_desc(xh + ko, kLbo, kSbo),
                             tc::smem_desc(bh + ko, kLbo, kSbo), idesc, 1u);
                tc::mma_tf32(d, tc::smem_desc(xh + ko, kLbo, kSbo),
                             tc::smem_desc(bl + ko, kLbo, kSbo), idesc, 1u);
                tc::mma_tf32(d, tc::smem_desc(xl + ko, kLbo, kSbo),
                             tc::smem_desc(bh + ko, kLbo, kSbo), idesc, 1u);
            }
        }
        if constexpr (FUSED) {
            if (tid == 0) {
                // D += X_j X_j^T (M = N = 128, K = 32); the cross terms in the
                // order that makes the upper storage's D the transpose, bit for
                // bit, of the lower storage's
                const uint32_t xh = sbase + kOffX, xl = xh + kXTile;
                const uint32_t p2a = UP ? xl : xh, p2b = UP ? xh : xl;
                const uint32_t p3a = UP ? xh : xl, p3b = UP ? xl : xh;
                constexpr uint32_t idesc = tc::idesc_tf32(128, 128);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t ko = ks * 2 * kLbo;
                    tc::mma_tf32(tmem + 128, tc::smem_desc(xh + ko, kLbo, kSbo),
                                 tc::smem_desc(xh + ko, kLbo, kSbo), idesc,
                                 (j > 0 || ks > 0) ? 1u : 0u);
                    tc::mma_tf32(tmem + 128, tc::smem_desc(p2a + ko, kLbo, kSbo),
                                 tc::smem_desc(p2b + ko, kLbo, kSbo), idesc, 1u);
                    tc::mma_tf32(tmem + 128, tc::smem_desc(p3a + ko, kLbo, kSbo),
                                 tc::smem_desc(p3b + ko, kLbo, kSbo), idesc, 1u);
                }
            }
        }
        if (tid == 0) {
            tc::mma_commit(&mbar);
            pend = j;
        }
    }

    if constexpr (FUSED) {
        // the last group's completion (the fourth commit), then
        // A22 -= D on the lower triangle of L's trailing block: thread r holds
        // D's row r; lower storage: it updates the entries (r, c), c <= r,
        // coalesced over r; upper storage: the entries (c, r), c >= r, whose
        // memory (c1 + r) + (c1 + c) lda is coalesced over r too
        if (tid == 0 && !sh_err) {
            if (tc::mbar_wait(&mbar, 1, kWaitCycles)) pend = -1;
            else sh_err = 1;
        }
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        const int m = n - c0 - 128, r = tid, c1 = c0 + 128;
        if (!sh_err) {  // uniform: the tensor-memory loads are warp-wide
            float *Cr = Ab + (int64_t)c1 * lda + c1 + r;  // Cr[c * lda] = memory (c1 + r, c1 + c)
#pragma unroll 1
            for (int h = 0; h < 4; ++h) {
                float v[32], old[32];
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const int c = 32 * h + t;
                    const bool in = r < m && c < m && (UP ? c >= r : c <= r);
                    old[t] = in ? Cr[(int64_t)c * lda] : 0.0f;
                }
                tc::tmem_ld32(tlane + 128 + 32 * h, v);
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const int c = 32 * h + t;
                    const bool in = r < m && c < m && (UP ? c >= r : c <= r);
                    if (in) Cr[(int64_t)c * lda] = old[t] - v[t];
                }
            }
        }
    }

    // a block that gave up lets its last MMA group drain (bounded) first: no
    // MMA may still write the tensor memory it releases
    if (tid == 0 && sh_err && pend >= 0) tc::mbar_wait(&mbar, pend & 1, kWaitCycles);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kCols);
    if (tid == 0 && sh_err) info[mat] = -1;
}

// The fused form keeps three blocks per SM although three 256-column
// accumulators exceed the SM's 512 columns: the third block's allocation
// waits for one of the others to finish (measured: 4096 matrices of order 200
// 771 us, against 780 us with two blocks per SM)
constexpr int kSmemFused = kSmemBytes;

template <bool UP, bool FUSED>
int launch_k(float *A, int n, int lda, int64_t strideA, int batch, int *info, int c0,
             cudaStream_t stream)
{
    constexpr int smem = FUSED ? kSmemFused : kSmemBytes;
    static DeviceOnce attrs;
    if (const int e = attrs.run([] {
            return cudaFuncSetAttribute(trsm_tc_kernel<UP, FUSED>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        }))
        return e;
    const int m = n - c0 - 128;
    const int nrb = (m + 127) / 128;
    const int64_t blocks = (int64_t)batch * nrb;
    if (blocks > 0x7fffffffLL) return (int)cudaErrorInvalidConfiguration;
    return launch_pdl(trsm_tc_kernel<UP, FUSED>, dim3((unsigned)blocks), dim3(128), (size_t)smem,
                      stream, A, n, lda, strideA, c0, nrb, info);
}

}  // namespace

int set_fail_first_wait_trsm_tc(int every)
{
    return (int)cudaMemcpyToSymbol(g_fail_first_wait, &every, sizeof every);
}

// Returns 0 after launching, 1 when the caller must use the FP32 kernel
// (unaligned panels), or a cudaError_t.
int launch_trsm_tc(float *A, int n, int lda, int64_t strideA, int batch, int *info, int c0,
                   cudaStream_t stream, bool upper, bool fused)
{
    if (((reinterpret_cast<uintptr_t>(A) & 15) != 0) || (lda & 3) || (strideA & 3)) return 1;
    if (fused && n - c0 - 128 > 128) return -1;
    if (fused)
        return upper ? launch_k<true, true>(A, n, lda, strideA, batch, info, c0, stream)
                     : launch_k<false, true>(A, n, lda, strideA, batch, info, c0, stream);
    return upper ? launch_k<true, false>(A, n, lda, strideA, batch, info, c0, stream)
                 : launch_k<false, false>(A, n, lda, strideA, batch, info, c0, stream);
}

}  // namespace bl
