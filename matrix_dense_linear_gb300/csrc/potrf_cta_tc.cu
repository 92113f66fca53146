// K2c: batched SPOTRF for n = 128 with 16-byte aligned columns: K2 with the
// trailing update on the tensor cores.
//
// The lower triangle stays in shared memory in K2's packed panel layout, and
// the schedule is K2's right-looking one (32-column panels, one warp factors
// each diagonal block, one thread per row solves the panel below it, the
// trsm_panel kernel of "kernelbot-cholesky-930185"). What changes is the
// trailing update A22 <- A22 - L21 L21^T of each panel, the bulk of K2's
// instructions: every thread that solves a row of L21 also splits it into
// TF32 hi + lo (3xTF32, x = hi + lo with hi exact in TF32; hi*hi + hi*lo +
// lo*hi) and stores it as a K-major operand row; one thread issues
// tcgen05.mma with L21 as both operands, D = L21 L21^T accumulating in tensor
// memory; the warps then subtract D from the stored triangle - first the next
// panel's columns, then one warp factors the next diagonal block while the
// others subtract the remaining columns (K2's look-ahead).
//
// The MMA has M = 128 rows: the operand starts 32 rows (four core-matrix row
// groups) before the staged L21 rows, so TMEM lane m holds matrix row c0 + m
// and lanes 0..31 (and, for later panels, lanes past row 127) hold products
// of whatever precedes or follows the staged rows in shared memory - they are
// never read. Warp w may only read TMEM lanes 32w .. 32w+31, so warps 1..3
// own the epilogue rows and warp 0 or 1 (by block parity) factors the
// diagonal blocks. Every wait is bounded; a block that gives up marks
// info = -1.
#include <mutex>

#include "cta_common.cuh"

namespace bl {
namespace {

using namespace cta;

constexpr int kNB = 4, kNP = 128, kNT = 128;
using Gm = CtaGeom<kNB>;
constexpr uint32_t kLbo = 128;               // K-adjacent core matrices
constexpr uint32_t kSbo = 8 * 128 + 16;      // K = 32 per row group, +16 B (banks)
constexpr uint32_t kStageRows = 96;          // L21 of panel 0, the largest
constexpr uint32_t kStageTile = kStageRows / 8 * kSbo;
constexpr uint32_t kOffStage = (uint32_t)Gm::bytes;  // after the packed triangle
constexpr int kSmemBytes = (int)(kOffStage + 2 * kStageTile);
static_assert(Gm::bytes % 128 == 0, "operand tiles must stay 16-byte aligned");
static_assert(kOffStage >= 4 * kSbo, "the M = 128 operand reads four row groups before it");

__device__ __forceinline__ uint32_t core_off(int r, int q)
{
    return (uint32_t)(r >> 3) * kSbo + (uint32_t)q * kLbo + (uint32_t)(r & 7) * 16;
}

// S(row, c .. c+31) -= v, row and c in matrix coordinates, c a panel start
__device__ __forceinline__ void sub_chunk(float *S, int row, int c, const float (&v)[32])
{
    const int q = c >> 5;
    float *dst = S + Gm::off(q) + (row - c);  // element (row, c + k) at dst[k * ld(q)]
    const int ldq = Gm::ld(q);
#pragma unroll
    for (int k = 0; k < 32; ++k) dst[k * ldq] -= v[k];
}

__global__ void __launch_bounds__(kNT, 3)
potrf_cta_tc_kernel(float *__restrict__ A, int lda, int64_t strideA, int *__restrict__ info,
                    int info_off)
{
    extern __shared__ __align__(128) uint8_t smem[];
    float *S = reinterpret_cast<float *>(smem);
    uint8_t *stg = smem + kOffStage;  // hi tile, then lo tile
    __shared__ __align__(16) float colbuf[2][32];
    __shared__ __align__(16) float sinv[32];
    __shared__ __align__(8) uint64_t mbar[3];  // bulk loads (panel 0, the rest), MMA
    __shared__ uint32_t tmem_base;
    __shared__ int sh_fail, sh_err;

    const int64_t mat = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    if (info_off >= 0 && info[mat] != 0) return;  // failed at an earlier panel
    float *__restrict__ Ab = A + mat * strideA;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dwarp = (int)(blockIdx.x & 1);  // factors the diagonal blocks
    // the order as a run-time value: the diagonal factor's column loop then
    // keeps its exit test, which stops the compiler from hoisting work across
    // columns (register pressure)
    int n = kNP;
    asm volatile("" : "+r"(n));

    if (tid == 0) {
        sh_fail = 0;
        sh_err = 0;
        tc::mbar_init(&mbar[0], 32);
        tc::mbar_init(&mbar[1], kNP - 32);
        tc::mbar_init(&mbar[2], 1);
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

    bulk_load_full<kNB>(S, Ab, lda, tid, mbar);
    if (tid == 0 && !tc::mbar_wait(&mbar[0], 0, kWaitCycles)) sh_err = 1;
    __syncthreads();
    if (warp == dwarp && !sh_err)
        factor_diag_block(S, Gm::ld(0), lane, 0, n, colbuf, sinv, &sh_fail);
    if (tid == 0 && !sh_err && !tc::mbar_wait(&mbar[1], 0, kWaitCycles)) sh_err = 1;
    __syncthreads();

    const uint32_t sb = tc::smem_u32(stg);
    int mma_phase = 0, mma_pending = 0;
#pragma unroll 1
    for (int p = 0; p < kNB - 1 && !sh_fail && !sh_err; ++p) {
        const int c0 = 32 * p, c1 = c0 + 32;
        float *P = S + Gm::off(p);
        const int ldp = Gm::ld(p);
        const int nrows = kNP - c1;  // rows of L21 (= N of the MMA)

        // panel solve; each solved row becomes a K-major operand row (hi, lo)
        if (tid < nrows) {
            float x[32];
            trsm_row_x(P, ldp, 32 + tid, sinv, x);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float h[4], l[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) tc::split_tf32(x[4 * q + u], h[u], l[u]);
                const uint32_t off = core_off(tid, q);
                *reinterpret_cast<float4 *>(stg + off) = make_float4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<float4 *>(stg + kStageTile + off) =
                    make_float4(l[0], l[1], l[2], l[3]);
            }
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (tid == 0) {
            // D = L21 L21^T: M = 128 (rows c0 .. c0+127), N = nrows, K = 32
            const uint32_t N = (uint32_t)nrows;
            const uint32_t idesc = tc::idesc_tf32(128, N);
            const uint32_t bh = sb, bl = sb + kStageTile;
            const uint32_t ah = bh - 4 * kSbo, al = bl - 4 * kSbo;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint32_t ko = ks * 2 * kLbo;
                tc::mma_tf32(tmem, tc::smem_desc(ah + ko, kLbo, kSbo),
                             tc::smem_desc(bh + ko, kLbo, kSbo), idesc, ks > 0 ? 1u : 0u);
                tc::mma_tf32(tmem, tc::smem_desc(ah + ko, kLbo, kSbo),
                             tc::smem_desc(bl + ko, kLbo, kSbo), idesc, 1u);
                tc::mma_tf32(tmem, tc::smem_desc(al + ko, kLbo, kSbo),
                             tc::smem_desc(bh + ko, kLbo, kSbo), idesc, 1u);
            }
            tc::mma_commit(&mbar[2]);
        }
        mma_pending = 1;
        if (tid == 0 && !tc::mbar_wait(&mbar[2], mma_phase, kWaitCycles)) sh_err = 1;
        tc::fence_before_sync();
        __syncthreads();
        if (sh_err) break;
        tc::fence_after_sync();
        mma_pending = 0;
        mma_phase ^= 1;

        // warp w holds TMEM lanes 32w.. = matrix rows c0 + 32w + lane
        const int row = c0 + 32 * warp + lane;
        const bool rows_ok = warp >= 1 && c0 + 32 * warp < kNP;
        const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
        if (rows_ok) {  // the next panel's columns c1 .. c1+31
            float v[32];
            tc::tmem_ld32(tl, v);
            sub_chunk(S, row, c1, v);
        }
        __syncthreads();
        if (warp == dwarp) {
            factor_diag_block(S + Gm::off(p + 1), Gm::ld(p + 1), lane, c1, n, colbuf, sinv,
                              &sh_fail);
        } else if (rows_ok) {
            // columns c1 + 32t, t = 1 .. warp - 1: the blocks left of and on
            // this warp's diagonal block
            for (int t = 1; t < warp; ++t) {
                float v[32];
                tc::tmem_ld32(tl + 32 * t, v);
                sub_chunk(S, row, c1 + 32 * t, v);
            }
        }
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }

    if (sh_err) {
        // a load or an MMA never completed: report it, let anything still in
        // flight drain (bounded) before the memory is released
        if (tid == 0) {
            tc::mbar_wait(&mbar[0], 0, kWaitCycles);
            tc::mbar_wait(&mbar[1], 0, kWaitCycles);
            if (mma_pending) tc::mbar_wait(&mbar[2], mma_phase, kWaitCycles);
            info[mat] = -1;
        }
        tc::fence_before_sync();
        __syncthreads();
        if (warp == 0) tc::tmem_dealloc(tmem, 128);
        return;
    }
    if (warp == 0) tc::tmem_dealloc(tmem, 128);
    tc::fence_async_smem();
    __syncthreads();
    bulk_store_full<kNB>(S, Ab, lda, tid);
    if (tid == 0) {
        const int f = sh_fail;
        if (info_off < 0) info[mat] = f;
        else if (f) info[mat] = info_off + f;
    }
}

}  // namespace

// n = 128, A, lda and strideA 16-byte aligned (the caller checks).
int launch_cta_tc(float *A, int lda, int64_t strideA, int batch, int *info, cudaStream_t stream,
                  InfoMode mode)
{
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(potrf_cta_tc_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    });
    if (attr != cudaSuccess) return (int)attr;
    return launch_pdl(potrf_cta_tc_kernel, dim3((unsigned)batch), dim3(kNT),
                      (size_t)kSmemBytes, stream, A, lda, strideA, info, mode.off);
}

int attrs_cta_tc(cudaFuncAttributes *fa, int *threads, int *dyn_smem)
{
    *threads = kNT;
    *dyn_smem = kSmemBytes;
    return (int)cudaFuncGetAttributes(fa, potrf_cta_tc_kernel);
}

}  // namespace bl
