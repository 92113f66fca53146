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
#include "launch.cuh"
#include "tc_sm100.cuh"

namespace bl {
namespace {

// failure injection for the give-up test (see set_fail_first_wait in launch.cuh)
__device__ int g_fail_first_wait;

constexpr uint32_t kLbo = 128;               // K-adjacent core matrices
constexpr uint32_t kSbo = 8 * 128 + 16;      // K = 32 per row group, +16 B (banks)
constexpr uint32_t kTileBytes = 16 * kSbo;   // 128 rows
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
__host__ __device__ constexpr int pk_base(int p) { return 32 * (p * 128 - 32 * (p * (p - 1) / 2)); }
__host__ __device__ constexpr int pk_ld(int p) { return 128 - 32 * p; }

__global__ void __launch_bounds__(128, 4)
potrf_tmem_kernel(float *__restrict__ A, int n, int lda, int64_t strideA, int batch,
                  int *__restrict__ info, int info_off)
{
    extern __shared__ __align__(128) uint8_t smem[];      // packed copy, then operand tiles
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
    const int NB = (n + 31) >> 5;
    // Row and column blocks are rotated against the TMEM lane quarters and
    // column blocks by rot: matrix block b lives in quarter / column block
    // (b + rot) % 4. Warp w (which may only address lane quarter w, and runs
    // on SM sub-partition w) therefore holds matrix row block (w - rot) % 4,
    // and the warp that factors panel p changes from block to block, so the
    // serial diagonal factors of co-resident blocks do not queue on one
    // sub-partition. The operand tile rows follow the TMEM lanes, so both MMA
    // operands see the same permutation.
    const int rot = (int)(blockIdx.x & 3);
    const int rb = (warp - rot) & 3;   // this warp's matrix row block
    const int row = 32 * rb + lane;    // this thread's matrix row
    auto tcol = [rot](int b) { return 32 * ((b + rot) & 3); };  // TMEM column of block b

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

    // -A into TMEM: copy the lower triangle into shared memory (column k by
    // one warp; 16-byte copies when aligned), then every thread moves its
    // row's chunks (column blocks 0 .. rb) into TMEM
    {
        float *S = reinterpret_cast<float *>(smem);
        const bool vec = ((reinterpret_cast<uintptr_t>(Ab) & 15) == 0) && ((lda & 3) == 0);
        for (int k = warp; k < n; k += 4) {
            const int pk = k >> 5;
            float *col = S + pk_base(pk) + (k - 32 * pk) * pk_ld(pk) - 32 * pk;  // col[r]
            const float *g = Ab + (int64_t)k * lda;
            int qa = n, qb = n;
            if (vec) {
                qa = (k + 3) & ~3;
                qb = n & ~3;
                if (qb < qa) qa = qb = n;
            }
            for (int q = qa + 4 * lane; q < qb; q += 128) cp_async16(col + q, g + q);
            for (int r = k + lane; r < n; r += 32)
                if (r < qa || r >= qb) cp_async4(col + r, g + r);
        }
        cp_async_commit();
        cp_async_wait<0>();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        const uint32_t tlane0 = tmem_base + ((uint32_t)(32 * warp) << 16);
        const int nch = min(rb, NB - 1) + 1;
#pragma unroll 1
        for (int j = 0; j < nch; ++j) {
            const float *src = S + pk_base(j) + (row - 32 * j);  // element (row, 32j + c)
            const int ldj = pk_ld(j);
            float v[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const int col = 32 * j + c;
                float x = (row == col) ? -1.0f : 0.0f;
                if (row < n && col <= row) x = -src[c * ldj];
                v[c] = x;
            }
            tc::tmem_st32(tlane0 + tcol(j), v);
        }
    }
    tc::fence_before_sync();
    __syncthreads();  // the shared copy is dead from here on (operand tiles reuse it)
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base;
    const uint32_t tlane = tmem + ((uint32_t)(32 * warp) << 16);

    // Trailing update of panel p: group 0 (mbar[0]) updates the next panel's
    // 32 columns, which the next panel waits for; group 1 (mbar[1]) the
    // columns after those, waited for only before the operand tile is
    // overwritten - the next diagonal factor runs while it is still on the
    // tensor cores. One MMA chain of N = 32 per column block. One thread waits
    // on an mbarrier; the others sleep at the block barrier.
    const uint32_t sbase = tc::smem_u32(smem);
    int n0 = 0, n1 = 0;  // commits to mbar[0] / mbar[1] so far (same in every thread)
#pragma unroll 1
    for (int p = 0; p < NB; ++p) {
        const int c0 = 32 * p;
        if (p > 0) {
            if (tid == 0 && ((p == 1 && injected_failure(g_fail_first_wait, mat)) ||
                             !tc::mbar_wait(&mbar[0], (n0 - 1) & 1, kWaitCycles)))
                sh_err = 1;
            tc::fence_before_sync();
            __syncthreads();
            if (sh_err) break;
            tc::fence_after_sync();
        }
        float x[32];
        if (rb >= p) {
            tc::tmem_ld32(tlane + tcol(p), x);
#pragma unroll
            for (int k = 0; k < 32; ++k) x[k] = -x[k];
        }
        if (rb == p) {
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
            if (row < n) {
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    if (k < lane) Ab[row + (int64_t)(c0 + k) * lda] = x[k];
                Ab[row + (int64_t)row * lda] = sqrt_approx(dm);
            }
            const unsigned bad = __ballot_sync(0xffffffffu, row < n && !pivot_ok(dm));
            if (lane == 0 && bad) sh_fail = c0 + __ffs(bad);
        }
        __syncthreads();
        if (sh_fail) break;
        if (rb > p) {
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
        // operand tile (row = TMEM lane): rows of blocks > p carry L21 split hi /
        // lo, the rest zeros
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float h[4], l[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                if (rb > p) tc::split_tf32(x[4 * q + t], h[t], l[t]);
                else h[t] = l[t] = 0.0f;
            }
            const uint32_t off = core_off(tid, q);
            *reinterpret_cast<float4 *>(smem + off) = make_float4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<float4 *>(smem + kTileBytes + off) =
                make_float4(l[0], l[1], l[2], l[3]);
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        // -S[:, block b] += L21 L21[block b, :]^T for b = p+1 .. NB-1 (M = 128, N = 32)
        const bool rest = p + 2 < NB;
        if (tid == 0) {
            const uint32_t a_hi = sbase, a_lo = sbase + kTileBytes;
            const uint32_t idesc = tc::idesc_tf32(128, 32);
#pragma unroll 1
            for (int b = p + 1; b < NB; ++b) {
                const uint32_t tc_b = (uint32_t)tcol(b);
                const uint32_t boff = (tc_b >> 3) * kSbo;  // tile rows of row block b
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t ko = ks * 2 * kLbo;
                    tc::mma_tf32(tmem + tc_b, tc::smem_desc(a_hi + ko, kLbo, kSbo),
                                 tc::smem_desc(a_hi + boff + ko, kLbo, kSbo), idesc, 1u);
                    tc::mma_tf32(tmem + tc_b, tc::smem_desc(a_hi + ko, kLbo, kSbo),
                                 tc::smem_desc(a_lo + boff + ko, kLbo, kSbo), idesc, 1u);
                    tc::mma_tf32(tmem + tc_b, tc::smem_desc(a_lo + ko, kLbo, kSbo),
                                 tc::smem_desc(a_hi + boff + ko, kLbo, kSbo), idesc, 1u);
                }
                if (b == p + 1) tc::mma_commit(&mbar[0]);
            }
            if (rest) tc::mma_commit(&mbar[1]);
        }
        ++n0;
        if (rest) ++n1;
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

DeviceOnce g_attrs;

}  // namespace

int set_fail_first_wait_tmem(int every)
{
    return (int)cudaMemcpyToSymbol(g_fail_first_wait, &every, sizeof every);
}

int launch_tmem(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                cudaStream_t stream, InfoMode mode)
{
    if (const int e = g_attrs.run([] {
            return cudaFuncSetAttribute(potrf_tmem_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        }))
        return e;
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
