// K2: batched SPOTRF for n <= 128, one thread block per matrix, the lower
// triangle resident in shared memory for the whole factorization.
//
// Storage. The padded order NP = 32*NB is split into NB block columns
// ("panels") of 32 columns. Panel p keeps only its rows 32p .. NP-1, as a
// column-major (NP-32p) x 32 rectangle with leading dimension NP-32p+4 (the
// +4 keeps 16-byte alignment and shifts banks between columns). The whole
// lower triangle then costs NP(NP+32)/2 floats: 43 KB at n = 128.
//
// Schedule (right-looking, one panel per step, after the inner-blocked
// schedule of "kernelbot-cholesky-930185", chol_diag_b kernel comment: the
// barriers, not the FMAs, are the critical path, so spend work to save them):
//   1. one warp factors the 32 x 32 diagonal block alone, lane = row, with the
//      same broadcast-column step as K1 (no block barrier inside); which warp
//      rotates with the panel and the block index, so the serial factors of
//      co-resident blocks spread over the SM's four sub-partitions;
//   2. every thread solves one row of the panel below it against that block,
//      P <- P L11^{-T}, reading L11's columns as 16-byte broadcasts
//      (the trsm_panel kernel of the same page: one thread per row);
//   3. every thread updates 4 x 4 tiles of the trailing LOWER triangle only,
//      A22 <- A22 - L21 L21^T (the page's left-looking driver note measured a
//      full-square trailing update as doubling the flops): first the next
//      panel's columns, then (look-ahead) one warp factors the next diagonal
//      block while the other warps update the remaining columns;
// with one __syncthreads after each phase. Rows and columns n .. NP-1 are an
// identity block. The upper storage (uplo = 'U') only changes the load and
// the store: row c of L is copied from / to column c of the upper triangle. Entries above the diagonal inside a diagonal block of the
// storage are scratch: they are never read into a lower result or stored.
#include <mutex>

#include "cta_common.cuh"
#include "launch.cuh"

namespace bl {
namespace {

using namespace cta;

// failure injection for the give-up test (see set_fail_first_wait in launch.cuh)
__device__ int g_fail_first_wait;

// Step 3: one 4 x 4 tile (I, K), I >= K, of the trailing lower triangle that
// starts at c1 = c0 + 32; L21 is panel p's rows c1.. . Pairs of rows go through
// the paired single-precision FMA (two fused multiply-adds, each rounded as
// fmaf, in one instruction).
template <int NB>
__device__ __forceinline__ void syrk_tile(float *S, const float *P, int ldp, int c0, int c1,
                                          int I, int K)
{
    using Gm = CtaGeom<NB>;
    const int gi = c1 + 4 * I, gk = c1 + 4 * K;
    const int q = gk >> 5;
    const int ldq = Gm::ld(q);
    float *C = S + Gm::off(q) + (gi - 32 * q) + (gk - 32 * q) * ldq;
    float2 acc[4][2];  // acc[b][h]: rows 2h, 2h + 1 of tile column b
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const float4 c4 = *reinterpret_cast<const float4 *>(C + b * ldq);
        acc[b][0] = make_float2(c4.x, c4.y); acc[b][1] = make_float2(c4.z, c4.w);
    }
    const float *Li = P + (gi - c0);
    const float *Lk = P + (gk - c0);
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
        const float4 a4 = *reinterpret_cast<const float4 *>(Li + k * ldp);
        const float4 b4 = *reinterpret_cast<const float4 *>(Lk + k * ldp);
        const float2 ap[2] = {make_float2(a4.x, a4.y), make_float2(a4.z, a4.w)};
        const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float2 nb = make_float2(-bv[b], -bv[b]);
#pragma unroll
            for (int h = 0; h < 2; ++h) acc[b][h] = __ffma2_rn(nb, ap[h], acc[b][h]);
        }
    }
#pragma unroll
    for (int b = 0; b < 4; ++b)
        *reinterpret_cast<float4 *>(C + b * ldq) =
            make_float4(acc[b][0].x, acc[b][0].y, acc[b][1].x, acc[b][1].y);
}

__device__ __forceinline__ void tri_index(int t, int &I, int &K)
{
    int i = (int)((sqrtf(8.0f * (float)t + 1.0f) - 1.0f) * 0.5f);
    while ((i + 1) * (i + 2) / 2 <= t) ++i;
    while (i * (i + 1) / 2 > t) --i;
    I = i;
    K = t - i * (i + 1) / 2;
}

// Copy columns [k0, k1) of the lower triangle (rows k .. n-1) into the
// packed storage; rows n .. NP-1 of those columns get the identity block.
template <int NB, int NT>
__device__ __forceinline__ void load_columns(float *S, const float *Ab, int n, int lda, int k0,
                                             int k1, bool vec, int warp, int lane)
{
    constexpr int NP = CtaGeom<NB>::NP;
    for (int k = k0 + warp; k < k1; k += NT / 32) {
        float *col = elem_ptr<NB>(S, 0, k);  // col[i] = element (i, k)
        const float *g = Ab + (int64_t)k * lda;
        const int lo = k, hi = k < n ? n : k;  // rows [lo, hi) come from memory
        int qa = hi, qb = hi;                   // rows [qa, qb) by 16-byte copies
        if (vec) {
            qa = (lo + 3) & ~3;
            qb = hi & ~3;
            if (qb < qa) qa = qb = hi;
        }
        for (int q = qa + 4 * lane; q < qb; q += 128) cp_async16(col + q, g + q);
        for (int i = lo + lane; i < hi; i += 32)
            if (i < qa || i >= qb) cp_async4(col + i, g + i);
        for (int i = hi + lane; i < NP; i += 32) col[i] = (i == k) ? 1.0f : 0.0f;
    }
}

// Store the lower triangle (rows < n) back, 16 bytes at a time where aligned.
template <int NB, int NT>
__device__ __forceinline__ void store_columns(const float *S, float *Ab, int n, int lda,
                                              bool vec, int warp, int lane)
{
    for (int k = warp; k < n; k += NT / 32) {
        const float *col = elem_ptr<NB>(const_cast<float *>(S), 0, k);
        float *g = Ab + (int64_t)k * lda;
        int qa = n, qb = n;
        if (vec) {
            qa = (k + 3) & ~3;
            qb = n & ~3;
            if (qb < qa) qa = qb = n;
        }
        for (int q = qa + 4 * lane; q < qb; q += 128)
            *reinterpret_cast<float4 *>(g + q) = *reinterpret_cast<const float4 *>(col + q);
        for (int i = k + lane; i < n; i += 32)
            if (i < qa || i >= qb) g[i] = col[i];
    }
}

// Upper storage (uplo = 'U'): row c of L is the contiguous column c of the
// upper triangle in memory (l_ck at Ab[k + c lda], k <= c). Rows c >= k0 of
// columns [k0, k1) are copied by warp c mod NW, lanes over k (coalesced 4-byte
// reads, each element to its place in the packed columns); then the identity
// rows of those columns as in load_columns.
template <int NB, int NT>
__device__ __forceinline__ void load_upper(float *S, const float *Ab, int n, int lda, int k0,
                                           int k1, int warp, int lane)
{
    constexpr int NP = CtaGeom<NB>::NP;
    for (int c = k0 + warp; c < n; c += NT / 32) {
        const float *g = Ab + (int64_t)c * lda;
        const int kend = c + 1 < k1 ? c + 1 : k1;
        for (int k = k0 + lane; k < kend; k += 32) cp_async4(elem_ptr<NB>(S, c, k), g + k);
    }
    for (int k = k0 + warp; k < k1; k += NT / 32) {
        float *col = elem_ptr<NB>(S, 0, k);
        const int hi = k < n ? n : k;
        for (int i = hi + lane; i < NP; i += 32) col[i] = (i == k) ? 1.0f : 0.0f;
    }
}

template <int NB, int NT>
__device__ __forceinline__ void store_upper(const float *S, float *Ab, int n, int lda, int warp,
                                            int lane)
{
    for (int c = warp; c < n; c += NT / 32) {
        float *g = Ab + (int64_t)c * lda;
        for (int k = lane; k <= c; k += 32) g[k] = *elem_ptr<NB>(const_cast<float *>(S), c, k);
    }
}

// FULL: n == NP and 16-byte aligned columns (the launcher checks): bulk copies.
// At n = 128 a thread gets 128 registers and four blocks share an SM: measured
// on GB300 that beats five blocks at 96 registers (60 against 67 us for 1024
// matrices).
// UP: the factor lives in the upper triangle (never with FULL).
template <int NB, int NT, bool FULL, bool UP>
__global__ void __launch_bounds__(NT, NB >= 3 ? 4 : 8)
potrf_cta_kernel(float *__restrict__ A, int n, int lda, int64_t strideA, int batch,
                 int *__restrict__ info, int info_off)
{
    using Gm = CtaGeom<NB>;
    constexpr int NP = Gm::NP;
    extern __shared__ __align__(16) float S[];
    __shared__ __align__(16) float colbuf[2][32];
    __shared__ __align__(16) float sinv[32];
    __shared__ __align__(8) uint64_t mbar[2];  // bulk loads: panel 0, the rest
    __shared__ int sh_fail, sh_err;

    const int64_t mat = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    if (info_off >= 0 && info[mat] != 0) return;  // failed at an earlier panel
    float *__restrict__ Ab = A + mat * strideA;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    // Load. 16-byte aligned batches (A, lda and strideA multiples of 4 floats)
    // of exact order n = NP take the bulk-copy path (one copy per column, all
    // in flight at once); otherwise column k is copied by one warp with
    // asynchronous 16-byte copies where both sides are aligned and 4-byte ones
    // at the ragged ends, and rows n .. NP-1 get the identity block. Either
    // way panel 0 is the first group: it is factored while the rest arrives.
    const bool vec = ((reinterpret_cast<uintptr_t>(A) & 15) == 0) && ((lda & 3) == 0) &&
                     ((strideA & 3) == 0);
    if (tid == 0) {
        sh_fail = 0;
        sh_err = 0;
        if constexpr (FULL) {
            tc::mbar_init(&mbar[0], 32);
            if (NB > 1) tc::mbar_init(&mbar[1], NP - 32);
            tc::fence_mbar_init();
        }
    }
    __syncthreads();
    if constexpr (FULL) {
        bulk_load_full<NB>(S, Ab, lda, tid, mbar);
        if (tid == 0 && (injected_failure(g_fail_first_wait, mat) ||
                         !tc::mbar_wait(&mbar[0], 0, kWaitCycles)))
            sh_err = 1;
    } else if constexpr (UP) {
        load_upper<NB, NT>(S, Ab, n, lda, 0, 32, warp, lane);
        cp_async_commit();
        load_upper<NB, NT>(S, Ab, n, lda, 32, NP, warp, lane);
        cp_async_commit();
        cp_async_wait<1>();
    } else {
        load_columns<NB, NT>(S, Ab, n, lda, 0, 32, vec, warp, lane);
        cp_async_commit();
        load_columns<NB, NT>(S, Ab, n, lda, 32, NP, vec, warp, lane);
        cp_async_commit();
        cp_async_wait<1>();
    }
    __syncthreads();

    // Panel 0's diagonal block, then per panel p (look-ahead): the panel solve
    // of p; the trailing update of the next panel's 32 columns; then warp 0
    // factors the next diagonal block while the other warps update the rest
    // of the trailing triangle (columns the next panel solve does not read).
    // The warp that factors a diagonal block rotates with the panel and the
    // block index: a warp runs on SM sub-partition (warp % 4), and a fixed
    // choice would queue the serial factor of every co-resident block on the
    // same sub-partition.
    constexpr int NW = NT / 32;
    const int rot = (int)(blockIdx.x % NW);
    if (warp == rot && !sh_err) factor_diag_block(S, Gm::ld(0), lane, 0, n, colbuf, sinv, &sh_fail);
    __syncthreads();
#pragma unroll 1
    for (int p = 0; p < NB && !sh_fail && !sh_err; ++p) {
        const int c0 = 32 * p;
        const int c1 = c0 + 32;
        if (c1 >= n) break;
        float *P = S + Gm::off(p);
        const int ldp = Gm::ld(p);
        for (int a = 32 + tid; a < NP - c0; a += NT) trsm_row(P, ldp, a, sinv);
        if (p == 0) {  // the trailing columns have arrived
            if constexpr (!FULL) cp_async_wait<0>();
            else if (tid == 0 && !tc::mbar_wait(&mbar[1], 0, kWaitCycles)) sh_err = 1;
        }
        __syncthreads();
        if (sh_err) break;
        // 4 x 4 tiles of the trailing triangle (rows/cols from c1), T per side;
        // consecutive threads take consecutive tile rows of one tile column
        const int T = (NP - c1) / 4;
        // the next panel's columns: tile columns 0..7, every tile row below
        for (int t = tid; t < 8 * T; t += NT) {
            const int K = t / T, I = t - K * T;
            if (I >= K) syrk_tile<NB>(S, P, ldp, c0, c1, I, K);
        }
        __syncthreads();
        const int dw = (p + 1 + rot) % NW;
        if (warp == dw) {
            factor_diag_block(S + Gm::off(p + 1), Gm::ld(p + 1), lane, c1, n, colbuf, sinv,
                              &sh_fail);
        } else {
            const int T2 = T - 8;  // tile columns 8 .. T-1, column-major order
            const int rank = (warp - dw - 1 + NW) % NW;  // among the other warps
            for (int t = 32 * rank + lane; t < T2 * (T2 + 1) / 2; t += NT - 32) {
                int a, b;
                tri_index(t, a, b);
                const int I = 8 + (T2 - 1 - b), K = 8 + (T2 - 1 - a);
                if (c1 + 4 * K < n) syrk_tile<NB>(S, P, ldp, c0, c1, I, K);
            }
        }
        __syncthreads();
    }

    if (sh_err) {
        // a bulk load never completed: report it, and give the copies a last
        // bounded chance to land before the shared memory is released
        if (tid == 0) {
            tc::mbar_wait(&mbar[0], 0, kWaitCycles);
            if (NB > 1) tc::mbar_wait(&mbar[1], 0, kWaitCycles);
            info[mat] = -1;
        }
        return;
    }
    if constexpr (FULL) {
        // a failed panel 0 leaves the loop before the second wait
        if (NB > 1 && tid == 0 && !tc::mbar_wait(&mbar[1], 0, kWaitCycles)) sh_err = 1;
        tc::fence_async_smem();  // this thread's shared-memory writes -> bulk stores
        __syncthreads();
        if (sh_err) {
            if (tid == 0) info[mat] = -1;
            return;
        }
        bulk_store_full<NB>(S, Ab, lda, tid);
    } else {
        cp_async_wait<0>();  // a failed panel 0 leaves the loop before the first wait
        __syncthreads();
        if constexpr (UP) store_upper<NB, NT>(S, Ab, n, lda, warp, lane);
        else store_columns<NB, NT>(S, Ab, n, lda, vec, warp, lane);
    }
    if (tid == 0) {
        const int f = sh_fail;
        if (info_off < 0) info[mat] = f;
        else if (f) info[mat] = info_off + f;
    }
}

template <int NB, int NT, bool FULL, bool UP>
int launch_v(float *A, int n, int lda, int64_t strideA, int batch, int *info, cudaStream_t st,
             int info_off)
{
    constexpr int bytes = CtaGeom<NB>::bytes;
    static DeviceOnce attrs;
    if (const int e = attrs.run([] {
            return cudaFuncSetAttribute(potrf_cta_kernel<NB, NT, FULL, UP>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        }))
        return e;
    return launch_pdl(potrf_cta_kernel<NB, NT, FULL, UP>, dim3((unsigned)batch), dim3(NT),
                      (size_t)bytes, st, A, n, lda, strideA, batch, info, info_off);
}

template <int NB, int NT>
int launch_nb(float *A, int n, int lda, int64_t strideA, int batch, int *info, cudaStream_t st,
              int info_off, bool upper, bool no_bulk)
{
    if (upper) return launch_v<NB, NT, false, true>(A, n, lda, strideA, batch, info, st, info_off);
    const bool vec = ((reinterpret_cast<uintptr_t>(A) & 15) == 0) && ((lda & 3) == 0) &&
                     ((strideA & 3) == 0);
    if (vec && n == CtaGeom<NB>::NP && !no_bulk)
        return launch_v<NB, NT, true, false>(A, n, lda, strideA, batch, info, st, info_off);
    return launch_v<NB, NT, false, false>(A, n, lda, strideA, batch, info, st, info_off);
}

// the n = NP bulk-copy kernel (the one the n = 128 and blocked workloads run)
template <int NB, int NT>
int attrs_nb(cudaFuncAttributes *fa, int *threads, int *dyn)
{
    *threads = NT;
    *dyn = CtaGeom<NB>::bytes;
    return (int)cudaFuncGetAttributes(fa, potrf_cta_kernel<NB, NT, true, false>);
}

}  // namespace

int set_fail_first_wait_cta(int every)
{
    return (int)cudaMemcpyToSymbol(g_fail_first_wait, &every, sizeof every);
}

int launch_cta(float *A, int n, int lda, int64_t strideA, int batch, int *info,
               cudaStream_t stream, InfoMode mode, bool upper, bool no_bulk)
{
    const int o = mode.off;
    const bool nb = no_bulk;
    // 64 < n <= 128, a whole matrix or a diagonal block of the blocked route
    // (info_off >= 0: its ragged last block, or unaligned batches): a warp per
    // 32 x 32 tile (potrf_tiles.cu) wherever the bulk-copy form below cannot run; 1024
    // matrices: n = 65 34.6 against 45.5 us, 112 70.8 against 86.1, 127 74.8
    // against 83.4; the bulk-copy form keeps n = 96 (36.7 against 42.0) and
    // 128 (58.7 against 74.6). The choice ignores no_bulk and uplo (the tile
    // kernel makes plain loads, fine on host-mapped memory, and reads either
    // storage), so a host batch gets the same kernel as on the device and the
    // upper storage the same arithmetic as the lower: the same bits.
    if (n > 64) {
        const bool vec = ((reinterpret_cast<uintptr_t>(A) & 15) == 0) && ((lda & 3) == 0) &&
                         ((strideA & 3) == 0);
        if (!(vec && (n == 96 || n == 128)))
            return launch_spotrf_tiles(A, n, lda, strideA, batch, info, stream, upper, o);
    }
    if (n <= 32) return launch_nb<1, 32>(A, n, lda, strideA, batch, info, stream, o, upper, nb);
    if (n <= 64) return launch_nb<2, 64>(A, n, lda, strideA, batch, info, stream, o, upper, nb);
    if (n <= 96) return launch_nb<3, 128>(A, n, lda, strideA, batch, info, stream, o, upper, nb);
    return launch_nb<4, 128>(A, n, lda, strideA, batch, info, stream, o, upper, nb);
}

// the kernel route 2 runs for this n on an aligned batch
int attrs_cta(int n, cudaFuncAttributes *fa, int *threads, int *dyn_smem)
{
    if (n > 64 && n != 96 && n != 128) return attrs_tiles(n, fa, threads, dyn_smem);
    if (n <= 32) return attrs_nb<1, 32>(fa, threads, dyn_smem);
    if (n <= 64) return attrs_nb<2, 64>(fa, threads, dyn_smem);
    if (n <= 96) return attrs_nb<3, 128>(fa, threads, dyn_smem);
    return attrs_nb<4, 128>(fa, threads, dyn_smem);
}

}  // namespace bl
