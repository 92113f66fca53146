// Trailing update of the blocked path on the tensor cores:
//     A22 <- A22 - L21 L21^T     (lower triangle, 128 x 128 output tiles, K = 128
//                                 or 256: one panel or two panels at once)
// with an error-compensated "3xTF32" split of the FP32 operands: each operand
// x = hi + lo with hi exact in TF32 and lo the FP32 remainder, and
//     L_I L_K^T ~= hi_I hi_K^T + hi_I lo_K^T + lo_I hi_K^T
// (the lo*lo term is below FP32 rounding). This is the trailing update the
// left-looking and blocked drivers of "kernelbot-cholesky-930185" ran through
// cuBLAS with TF32 (its notes record plain TF32 failing the reconstruction
// budget at n = 256); here it is a tcgen05 kernel of our own with the
// compensated split, the accumulator in tensor memory.
//
// One block (256 threads) per output tile (I, K), I >= K. The k dimension goes
// through shared memory 16 columns at a time in a ring of three buffers: every thread
// loads a 4 x 4 block of one operand (4 columns x 4 rows, 16-byte loads along
// the contiguous rows), splits it and writes it K-major (row r: k..k+3) into
// the hi and lo tiles; thread 0 then issues 2 k-steps x 3 products of
// tcgen05.mma (M = N = 128, K = 8) and commits them to the buffer's mbarrier;
// thread 0 alone waits on it, one slice ahead of the buffer's reuse, and the
// block barrier each slice has anyway passes that on. The next slice's global
// loads are in flight while the current one is written. The epilogue reads the
// accumulator back from tensor memory (warp w: rows 32(w%4).., columns
// 64(w/4)..) and subtracts it from A22 in place, lower triangle only.
//
// Two panels at once (K = 256): the blocked driver may delay a panel's update
// of everything right of the next panel's columns and apply it together with
// the next panel's update, so that each trailing tile is read and written
// once for two panels. The next panel's own columns are updated alone first
// (`narrow`: the first tile column of the trailing matrix only), since its
// diagonal factor and panel solve need them.
//
// Every wait is bounded (about a second); a block that gives up marks the
// matrix with info = -1 and still releases its tensor memory. The upper
// storage (uplo = 'U') changes only the addresses: a row of L is contiguous
// there, so the 16-byte loads run along the rows and need no transpose.
#include <mutex>

#include "bl_common.cuh"
#include "launch.cuh"
#include "tc_sm100.cuh"

namespace bl {
namespace {

constexpr int kNbTc = 128;                 // panel width
constexpr int kKs = 16;                    // k columns per shared-memory slice
constexpr uint32_t kLbo = 144;             // K-adjacent core matrices, +16 B: the upper storage's
                                           // staging stores (a row's four k quads) on distinct banks
constexpr uint32_t kSbo = (kKs / 4) * kLbo + 16;  // row-group stride, +16 B: no bank conflicts
constexpr uint32_t kTileBytes = 16 * kSbo;  // 128 rows
constexpr uint32_t kStageBytes = 4 * kTileBytes;  // A hi, A lo, B hi, B lo
constexpr int kStages = 3;                 // operand buffers in the ring
constexpr int kSmemBytes = kStages * kStageBytes;
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s at 2 GHz

// failure injection for the give-up test (see set_fail_first_wait in launch.cuh)
__device__ int g_fail_first_wait;

__device__ __forceinline__ uint32_t core_off(int r, int kq)
{
    // byte offset of (row r, k = 4kq .. 4kq+3) in a K-major no-swizzle tile
    return (uint32_t)(r >> 3) * kSbo + (uint32_t)kq * kLbo + (uint32_t)(r & 7) * 16;
}

template <bool UP>
__global__ void __launch_bounds__(256, 2)
syrk_tc_kernel(float *__restrict__ A, int n, int lda, int64_t strideA, int c0, int nk,
               int narrow, int ntiles_col, int *__restrict__ info)
{
    // k columns c0 .. c0+nk-1 (nk = 128 or 256); the trailing matrix starts at
    // c1 = c0 + nk; narrow: tile column 0 only (K = 0). The grid is one
    // dimension, the tile index fastest: a matrix's tiles run together, so its
    // panel is read from memory once and from L2 by the other tiles (with the
    // matrix fastest, a round of tiles over a large batch streams more than L2
    // holds between two tiles of one matrix).
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint32_t tmem_base;
    __shared__ __align__(8) uint64_t mbar[kStages];
    __shared__ int sh_err;

    const int nt = narrow ? ntiles_col : ntiles_col * (ntiles_col + 1) / 2;  // tiles a matrix
    const int64_t mat = blockIdx.x / nt;
    const int tile = (int)(blockIdx.x % nt);
    // launched as a programmatic dependent: wait for the previous kernel's
    // writes, then let the next kernel of the stream start launching
    pdl_wait();
    pdl_trigger();
    if (block_skip(info, mat)) return;
    int I, K;
    if (narrow) {
        I = tile;
        K = 0;
    } else {
        const int t = tile;
        int i = (int)((sqrtf(8.0f * (float)t + 1.0f) - 1.0f) * 0.5f);
        while ((i + 1) * (i + 2) / 2 <= t) ++i;
        while (i * (i + 1) / 2 > t) --i;
        I = i;
        K = t - i * (i + 1) / 2;
    }
    float *__restrict__ Ab = A + mat * strideA;
    const int c1 = c0 + nk;
    const int m = n - c1;
    const int nslices = nk / kKs;
    const int ri = I * 128, rk = K * 128;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // The MMA computes D[r][c] = sum_k L(tm + r, k) L(tn + c, k). Lower storage:
    // (tm, tn) = (ri, rk), D is the tile itself. Upper storage: (tm, tn) =
    // (rk, ri), D is the tile's transpose, so that in both storages the
    // epilogue's element (r, c) lives at (c1 + tm + r) + (c1 + tn + c) lda: a
    // warp's 32 rows r are contiguous in memory.
    const int tm = UP ? rk : ri, tn = UP ? ri : rk;

    // this thread stages one 4 x 4 block of one operand per slice; lower: a
    // warp's lanes take 32 row quads (16-byte loads down a column), upper: 8
    // row quads x 4 k quads (16-byte loads along the rows, 64 bytes a row)
    const int op = tid >> 7;                            // 0: rows tm.. (A), 1: rows tn.. (B)
    // a diagonal tile's two operands are the same rows: staged once (op 0),
    // and the MMAs read that copy as B too
    const bool stager = !(op == 1 && tm == tn);
    const int rq = UP ? (tid >> 2) & 31 : tid & 31;     // row quad: rows 4rq .. 4rq+3
    const int kq = UP ? tid & 3 : (tid >> 5) & 3;       // k quad within the slice
    const int rbase = op ? tn : tm;
    const int mrows = m - rbase;        // rows of this operand that exist
    // lower storage: src[c * lda + i] = (row 4rq + i, k = 4kq + c), 16 bytes down
    // a column; upper storage: src[i * lda + c], 16 bytes along a row
    const float *src = Ab + lidx<UP>(c1 + rbase + 4 * rq, c0 + 4 * kq, lda);
    const int valid_rows = max(0, min(4, mrows - 4 * rq));

    if (tid == 0) {
        sh_err = 0;
        for (int i = 0; i < kStages; ++i) tc::mbar_init(&mbar[i], 1);
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
    const uint32_t sbase = tc::smem_u32(smem);
    constexpr uint32_t idesc = tc::idesc_tf32(128, 128);

    float4 cur[4], nxt[4], nxt2[4];  // lower: [k][4 rows]; upper: [row][4 k]
    auto load_slice = [&](int s, float4 (&v)[4]) {
        if (!stager) return;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if constexpr (UP) {
                const float *p = src + (int64_t)c * lda + s * kKs;
                v[c] = valid_rows > c ? *reinterpret_cast<const float4 *>(p)
                                      : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            } else {
                const float *p = src + (int64_t)(s * kKs + c) * lda;
                if (valid_rows == 4) {
                    v[c] = *reinterpret_cast<const float4 *>(p);
                } else {
                    v[c].x = valid_rows > 0 ? p[0] : 0.0f;
                    v[c].y = valid_rows > 1 ? p[1] : 0.0f;
                    v[c].z = valid_rows > 2 ? p[2] : 0.0f;
                    v[c].w = 0.0f;
                }
            }
        }
    };
    load_slice(0, cur);
    load_slice(1, nxt);

    const bool fail_first = injected_failure(g_fail_first_wait, mat);
    bool ok = true;
    int issued = 0;  // slices whose MMAs thread 0 has issued (same in every thread)
#pragma unroll 1
    for (int s = 0; s < nslices; ++s) {
        // a three-buffer ring: slice s goes to buffer s % 3, which the MMAs of
        // slice s - 3 read; thread 0 saw those complete before the previous
        // slice's barrier (below), so no thread waits here
        const int b = s % kStages;
        if (s + 2 < nslices) load_slice(s + 2, nxt2);  // two slices in flight
        // transpose the 4 x 4 block to K-major rows, split into hi and lo
        uint8_t *st = smem + b * kStageBytes + (op ? 2 : 0) * kTileBytes;
        const float cv[4][4] = {{cur[0].x, cur[0].y, cur[0].z, cur[0].w},
                                {cur[1].x, cur[1].y, cur[1].z, cur[1].w},
                                {cur[2].x, cur[2].y, cur[2].z, cur[2].w},
                                {cur[3].x, cur[3].y, cur[3].z, cur[3].w}};
#pragma unroll
        for (int i = 0; i < 4 && stager; ++i) {
            float h[4], l[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) tc::split_tf32(UP ? cv[i][c] : cv[c][i], h[c], l[c]);
            const uint32_t off = core_off(4 * rq + i, kq);
            *reinterpret_cast<float4 *>(st + off) = make_float4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<float4 *>(st + kTileBytes + off) = make_float4(l[0], l[1], l[2], l[3]);
        }
        tc::fence_async_smem();
        // the buffer the next slice overwrites is read by the MMAs of slice
        // s - 2: thread 0 alone waits for them, and the barrier tells the rest
        if (tid == 0 && s >= 2 &&
            ((s == 2 && fail_first) ||
             !tc::mbar_wait(&mbar[(s - 2) % kStages], ((s - 2) / kStages) & 1, kWaitCycles)))
            sh_err = 1;
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (sh_err) { ok = false; break; }
        if (tid == 0) {
            const uint32_t a_hi = sbase + b * kStageBytes, a_lo = a_hi + kTileBytes;
            const uint32_t b_hi = tm == tn ? a_hi : a_hi + 2 * kTileBytes;
            const uint32_t b_lo = b_hi + kTileBytes;
#pragma unroll
            for (int ks = 0; ks < kKs / 8; ++ks) {
                const uint32_t ko = ks * 2 * kLbo;
                const uint32_t acc0 = (s > 0 || ks > 0) ? 1u : 0u;
                // the cross terms in the order hi_I lo_K, lo_I hi_K in both
                // storages (the I side is A in the lower, B in the upper), so
                // both round alike
                const uint32_t x1a = UP ? a_lo : a_hi, x1b = UP ? b_hi : b_lo;
                const uint32_t x2a = UP ? a_hi : a_lo, x2b = UP ? b_lo : b_hi;
                tc::mma_tf32(tmem, tc::smem_desc(a_hi + ko, kLbo, kSbo),
                             tc::smem_desc(b_hi + ko, kLbo, kSbo), idesc, acc0);
                tc::mma_tf32(tmem, tc::smem_desc(x1a + ko, kLbo, kSbo),
                             tc::smem_desc(x1b + ko, kLbo, kSbo), idesc, 1u);
                tc::mma_tf32(tmem, tc::smem_desc(x2a + ko, kLbo, kSbo),
                             tc::smem_desc(x2b + ko, kLbo, kSbo), idesc, 1u);
            }
            tc::mma_commit(&mbar[b]);
        }
        ++issued;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            cur[c] = nxt[c];
            nxt[c] = nxt2[c];
        }
    }

    // this thread's 64 entries of A22 (its tile row, its column half) are
    // loaded while the last MMAs run
    // (gr, gc): trailing coordinates of D's row r and column c (lower: the
    // element (gr, gc) of L; upper: the element (gc, gr)); it lives at
    // Crow[gc * lda] either way, and is in the lower triangle of L when
    // gr >= gc (lower) or gc >= gr (upper)
    const int q = warp & 3, h = warp >> 2;
    const int r = 32 * q + lane;  // tile row
    const int gr = tm + r;        // trailing row
    const int gcb = tn + 64 * h;  // first trailing column of this half
    float *Crow = Ab + c1 + gr + (int64_t)c1 * lda;
    auto inside = [&](int gc) { return gr < m && gc < m && (UP ? gc >= gr : gr >= gc); };
    float old[32];  // the first two 16-column chunks; the other two follow
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int gc = gcb + j;
        old[j] = inside(gc) ? Crow[(int64_t)gc * lda] : 0.0f;
    }

    // all MMAs issued before the last commit are complete once it arrives; the
    // outcome is made block-uniform (tcgen05.ld is a warp-collective)
    const int last = issued - 1;
    if (tid == 0 && ok && !tc::mbar_wait(&mbar[last % kStages], (last / kStages) & 1, kWaitCycles))
        sh_err = 1;
    __syncthreads();
    ok = sh_err == 0;
    tc::fence_after_sync();

    const bool full = I != K && ri + 128 <= m && rk + 128 <= m;
    if (ok && full) {  // whole off-diagonal tile: no masks
        float *Cr = Crow + (int64_t)gcb * lda;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            if (half == 1) {
#pragma unroll
                for (int j = 0; j < 32; ++j) old[j] = Cr[(int64_t)(32 + j) * lda];
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float v[16];
                tc::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + 64 * h + 32 * half + 16 * c, v);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    Cr[(int64_t)(32 * half + 16 * c + j) * lda] = old[16 * c + j] - v[j];
            }
        }
    } else if (ok) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            if (half == 1) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int gc = gcb + 32 + j;
                    old[j] = inside(gc) ? Crow[(int64_t)gc * lda] : 0.0f;
                }
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float v[16];
                tc::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + 64 * h + 32 * half + 16 * c, v);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int gc = gcb + 32 * half + 16 * c + j;
                    if (inside(gc)) Crow[(int64_t)gc * lda] = old[16 * c + j] - v[j];
                }
            }
        }
    } else if (tid == 0) {
        info[mat] = -1;
        // let anything still in flight drain (bounded) before releasing TMEM
        if (last >= 0) tc::mbar_wait(&mbar[last % kStages], (last / kStages) & 1, kWaitCycles);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

template <bool UP>
int launch_u(float *A, int n, int lda, int64_t strideA, int batch, int *info, int c0, int nk,
             bool narrow, cudaStream_t stream)
{
    static DeviceOnce attrs;
    if (const int e = attrs.run([] {
            return cudaFuncSetAttribute(syrk_tc_kernel<UP>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        }))
        return e;
    const int m = n - c0 - nk;
    const int T = (m + 127) / 128;
    const int64_t blocks = (int64_t)batch * (narrow ? T : T * (T + 1) / 2);
    if (blocks > 0x7fffffffLL) return (int)cudaErrorInvalidConfiguration;
    return launch_pdl(syrk_tc_kernel<UP>, dim3((unsigned)blocks), dim3(256), (size_t)kSmemBytes,
                      stream, A, n, lda, strideA, c0, nk, narrow ? 1 : 0, T, info);
}

}  // namespace

int set_fail_first_wait_syrk_tc(int every)
{
    return (int)cudaMemcpyToSymbol(g_fail_first_wait, &every, sizeof every);
}

// Returns 0 and launches when the tensor-core path applies (16-byte aligned
// panels), 1 when the caller must use the FP32 path, or a cudaError_t.
int launch_syrk_tc(float *A, int n, int lda, int64_t strideA, int batch, int *info, int c0,
                   int nk, bool narrow, cudaStream_t stream, bool upper)
{
    if (((reinterpret_cast<uintptr_t>(A) & 15) != 0) || (lda & 3) || (strideA & 3)) return 1;
    if (nk <= 0 || nk % kKs != 0 || n - c0 - nk <= 0) return -1;
    return upper ? launch_u<true>(A, n, lda, strideA, batch, info, c0, nk, narrow, stream)
                 : launch_u<false>(A, n, lda, strideA, batch, info, c0, nk, narrow, stream);
}

int attrs_syrk_tc(cudaFuncAttributes *fa)
{
    return (int)cudaFuncGetAttributes(fa, syrk_tc_kernel<false>);
}

}  // namespace bl
