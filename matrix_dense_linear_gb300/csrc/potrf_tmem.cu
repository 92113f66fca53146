// K2t: batched SPOTRF for n <= 128 with the matrix resident in tensor memory.
//
// One block of 128 threads per matrix. Tensor memory (TMEM) holds the
// negated working matrix -S (S = the Schur complement still to be factored):
// lane r is row r, column c is column c, so warp w (which may only address
// lanes 32w .. 32w+31) owns rows 32w .. 32w+31 and one tcgen05.ld gives each of
// its lanes one row of a 32-column panel - the lane = row layout of the
// warp-level factorization. Per 32-column panel p (c0 = 32p):
//   1. warps >= p read their rows of the panel from TMEM;
//   2. warp p factors the 32 x 32 diagonal block in registers (the broadcast
//      column step of K1) and publishes L_pp and the reciprocal roots;
//   3. warps > p solve their rows against it (x <- x L_pp^{-T}, one row per
//      thread, the trsm_panel kernel of "kernelbot-cholesky-930185");
//   4. finished rows of the panel go straight to global memory;
//   5. the panel below the diagonal is split hi + lo (3xTF32) into a K-major
//      shared-memory tile and one thread issues 4 k-steps x 3 tcgen05.mma that
//      ADD L21 L21^T to -S in TMEM (= subtract it from S; no negated operands),
//      the trailing update of the right-looking schedule, lower part used.
// The only chain that remains on the SIMT side is the 32-step diagonal factor
// per panel; the trailing update runs on the tensor cores.
//
// Rows and columns n .. 127 are an identity block. info and the sub-block mode
// (used by the blocked path) are as in K2; a bounded wait that gives up marks
// info = -1.
#include <mutex>

#include "bl_common.cuh"
#include "tc_sm100.cuh"

namespace bl {
namespace {

constexpr uint32_t kLbo = 128;               // K-adjacent core matrices
constexpr uint32_t kSbo = 8 * 128 + 16;      // K = 32 per row group, +16 B (banks)
constexpr uint32_t kTileBytes = 16 * kSbo;   // 128 rows
constexpr int kOperandBytes = 2 * kTileBytes;  // hi, lo
// requested dynamic shared memory: the operand tiles, padded so that at most
// four blocks (4 x 128 TMEM columns = all 512) share an SM
constexpr int kSmemBytes = 48 * 1024;
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s

__device__ __forceinline__ uint32_t core_off(int r, int q)
{
    return (uint32_t)(r >> 3) * kSbo + (uint32_t)q * kLbo + (uint32_t)(r & 7) * 16;
}

// The lower triangle is first copied into shared memory in the packed panel
// layout of K2 (panel p keeps rows 32p .. 127 of its 32 columns, column-major,
// leading dimension 128 - 32p; 40 KB), every copy in flight at once.
__device__ __forceinline__ int pk_off(int r, int k)
{
    const int p = k >> 5;
    return 32 * (p * 128 - 32 * (p * (p - 1) / 2)) + (r - 32 * p) + (k - 32 * p) * (128 - 32 * p);
}

// 32 entries of row `row`, columns col0 .. col0+31, negated, from the packed
// copy (lower triangle of A; identity beyond n).
__device__ __forceinline__ void row_chunk(const float *S, int n, int row, int col0, float (&v)[32])
{
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        const int col = col0 + c;
        float x = (row == col) ? -1.0f : 0.0f;
        if (row < n && col <= row) x = -S[pk_off(row, col)];
        v[c] = x;
    }
}

__global__ void __launch_bounds__(128, 4)
potrf_tmem_kernel(float *__restrict__ A, int n, int lda, int64_t strideA, int batch,
                  int *__restrict__ info, int info_off)
{
    extern __shared__ __align__(128) uint8_t smem[];      // operand tiles: hi, lo
    __shared__ __align__(16) float Ls[32 * 32];            // Ls[j*32 + k] = L(c0+k, c0+j)
    __shared__ __align__(16) float colbuf[2][32];
    __shared__ __align__(16) float sinv[32];
    __shared__ uint32_t tmem_base;
    __shared__ __align__(8) uint64_t mbar[2];  // [0]: next panel's columns, [1]: the rest
    __shared__ int sh_fail, sh_err;

    const int64_t mat = blockIdx.x;
    if (info_off >= 0 && info[mat] != 0) return;  // failed at an earlier panel
    float *__restrict__ Ab = A + mat * strideA;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = tid;
    const int NB = (n + 31) >> 5;

    if (tid == 0) {
        sh_fail = 0;
        sh_err = 0;
        tc::mbar_init(&mbar[0], 1);
        tc::mbar_init(&mbar[1], 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, 128);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base;
    const uint32_t tlane = tmem + ((uint32_t)(32 * warp) << 16);

    // -A into TMEM: copy the lower triangle into shared memory (column k by
    // one warp), then warp w moves its rows' chunks 0 .. w into TMEM
    {
        float *S = reinterpret_cast<float *>(smem);
        for (int k = warp; k < n; k += 4) {
            const float *g = Ab + (int64_t)k * lda;
            for (int r = k + lane; r < n; r += 32) cp_async4(S + pk_off(r, k), g + r);
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        const int nch = min(warp, NB - 1) + 1;
#pragma unroll 1
        for (int j = 0; j < nch; ++j) {
            float v[32];
            row_chunk(S, n, row, 32 * j, v);
            tc::tmem_st32(tlane + 32 * j, v);
        }
    }
    tc::fence_before_sync();
    __syncthreads();  // the shared copy is dead from here on (operand tiles reuse it)
    tc::fence_after_sync();

    // Trailing update of panel p in two MMA groups: group 0 updates the next
    // panel's 32 columns and is committed to mbar[0] (the next panel waits only
    // for it), group 1 the columns after those, committed to mbar[1] (waited
    // for only before the operand tile is overwritten) - so the next diagonal
    // factor runs while the bulk of the update is still on the tensor cores.
    // One thread waits on an mbarrier; the others sleep at the block barrier.
    const uint32_t sbase = tc::smem_u32(smem);
    int n0 = 0, n1 = 0;  // commits to mbar[0] / mbar[1] so far (same in every thread)
#pragma unroll 1
    for (int p = 0; p < NB; ++p) {
        const int c0 = 32 * p;
        if (p > 0) {
            if (tid == 0 && !tc::mbar_wait(&mbar[0], (n0 - 1) & 1, kWaitCycles)) sh_err = 1;
            tc::fence_before_sync();
            __syncthreads();
            if (sh_err) break;
            tc::fence_after_sync();
        }
        float x[32];
        if (warp >= p) {
            tc::tmem_ld32(tlane + c0, x);
#pragma unroll
            for (int k = 0; k < 32; ++k) x[k] = -x[k];
        }
        if (warp == p) {
            // diagonal block: lane = row c0 + lane, columns c0 .. c0+31
            float dm = 1.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (c0 + j >= n) break;
                float *cb = colbuf[j & 1];
                cb[lane] = x[j];
                __syncwarp();
                const float d = cb[j];
                const float s = rsqrt_approx(d);
                const float l = x[j] * s;
                const float w = l * s;
                x[j] = l;
                dm = (lane == j) ? d : dm;
#pragma unroll
                for (int q = (j + 1) / 4; q < 8; ++q) {
                    const float4 c4 = reinterpret_cast<const float4 *>(cb)[q];
                    const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int k = 4 * q + t;
                        if (k > j) x[k] = fmaf(-w, cv[t], x[k]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < lane) Ls[j * 32 + lane] = x[j];
            sinv[lane] = rsqrt_approx(dm);
            const int r = c0 + lane;
            if (r < n) {
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    if (k < lane) Ab[r + (int64_t)(c0 + k) * lda] = x[k];
                Ab[r + (int64_t)r * lda] = sqrt_approx(dm);
            }
            const unsigned bad = __ballot_sync(0xffffffffu, r < n && !pivot_ok(dm));
            if (lane == 0 && bad) sh_fail = c0 + __ffs(bad);
        }
        __syncthreads();
        if (sh_fail) break;
        if (warp > p) {
            // x <- x L_pp^{-T}
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                x[j] *= sinv[j];
                const float *Lj = Ls + j * 32;
#pragma unroll
                for (int q = (j + 1) / 4; q < 8; ++q) {
                    const float4 l4 = reinterpret_cast<const float4 *>(Lj)[q];
                    const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int k = 4 * q + t;
                        if (k > j) x[k] = fmaf(-x[j], lv[t], x[k]);
                    }
                }
            }
            if (row < n) {
#pragma unroll
                for (int k = 0; k < 32; ++k) Ab[row + (int64_t)(c0 + k) * lda] = x[k];
            }
        }
        const int c1 = c0 + 32;
        if (c1 >= n) break;
        if (n1 > 0) {  // group 1 of the last panel still reads the operand tile
            if (tid == 0 && !tc::mbar_wait(&mbar[1], (n1 - 1) & 1, kWaitCycles)) sh_err = 1;
            __syncthreads();
            if (sh_err) break;
        }
        // operand tile: rows > c0+31 carry L21 (split hi / lo), the rest zeros
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float h[4], l[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                if (warp > p) tc::split_tf32(x[4 * q + t], h[t], l[t]);
                else h[t] = l[t] = 0.0f;
            }
            const uint32_t off = core_off(row, q);
            *reinterpret_cast<float4 *>(smem + off) = make_float4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<float4 *>(smem + kTileBytes + off) =
                make_float4(l[0], l[1], l[2], l[3]);
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        // -S[:, c:c+N] += L21 L21[c:c+N, :]^T  (M = 128 rows)
        const int nrest = 128 - c1 - 32;
        if (tid == 0) {
            const uint32_t a_hi = sbase, a_lo = sbase + kTileBytes;
#pragma unroll 1
            for (int g = 0; g < 2; ++g) {
                const int c = g == 0 ? c1 : c1 + 32;
                const uint32_t N = g == 0 ? 32u : (uint32_t)nrest;
                if (N == 0) break;
                const uint32_t idesc = tc::idesc_tf32(128, N);
                const uint32_t boff = (uint32_t)(c >> 3) * kSbo;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t ko = ks * 2 * kLbo;
                    tc::mma_tf32(tmem + c, tc::smem_desc(a_hi + ko, kLbo, kSbo),
                                 tc::smem_desc(a_hi + boff + ko, kLbo, kSbo), idesc, 1u);
                    tc::mma_tf32(tmem + c, tc::smem_desc(a_hi + ko, kLbo, kSbo),
                                 tc::smem_desc(a_lo + boff + ko, kLbo, kSbo), idesc, 1u);
                    tc::mma_tf32(tmem + c, tc::smem_desc(a_lo + ko, kLbo, kSbo),
                                 tc::smem_desc(a_hi + boff + ko, kLbo, kSbo), idesc, 1u);
                }
                tc::mma_commit(&mbar[g]);
            }
        }
        ++n0;
        if (nrest > 0) ++n1;
    }

    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {  // every issued MMA has completed before TMEM is released (bounded)
        if (n0 > 0 && !tc::mbar_wait(&mbar[0], (n0 - 1) & 1, kWaitCycles)) sh_err = 1;
        if (n1 > 0 && !tc::mbar_wait(&mbar[1], (n1 - 1) & 1, kWaitCycles)) sh_err = 1;
    }
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 128);
    if (tid == 0) {
        const int f = sh_fail;
        if (sh_err) info[mat] = -1;
        else if (info_off < 0) info[mat] = f;
        else if (f) info[mat] = info_off + f;
    }
}

std::once_flag g_once;
cudaError_t g_attr = cudaSuccess;

}  // namespace

int launch_tmem(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                cudaStream_t stream, InfoMode mode)
{
    std::call_once(g_once, [] {
        g_attr = cudaFuncSetAttribute(potrf_tmem_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    });
    if (g_attr != cudaSuccess) return (int)g_attr;
    potrf_tmem_kernel<<<(unsigned)batch, 128, kSmemBytes, stream>>>(A, n, lda, strideA, batch,
                                                                    info, mode.off);
    return (int)cudaGetLastError();
}

int attrs_tmem(int n, cudaFuncAttributes *fa, int *threads, int *dyn_smem)
{
    (void)n;
    *threads = 128;
    *dyn_smem = kSmemBytes;
    return (int)cudaFuncGetAttributes(fa, potrf_tmem_kernel);
}

}  // namespace bl
