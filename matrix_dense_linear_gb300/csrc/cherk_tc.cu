// Trailing update of the single-precision complex blocked path on the tensor
// cores (either storage; in the upper one an operand row is U's contiguous
// column and the raw values are L's conjugates, so the same products give the
// conjugated update the upper triangle stores):
//     A22 <- A22 - L21 L21^H      (lower triangle, 128 x 128 complex tiles, k = 128)
// in real arithmetic. With L = P + iQ (P, Q the real and imaginary parts),
//     L_I L_K^H = (P_I P_K^T + Q_I Q_K^T) + i (Q_I P_K^T - P_I Q_K^T),
// so each tile is two real accumulators in tensor memory (the real and the
// imaginary part, 128 columns each) and four real products, each taken in the
// error-compensated 3xTF32 form of syrk_tc.cu (x = hi + lo, hi exact in TF32:
// hi hi + hi lo + lo hi); the two products that are subtracted use the MMA's
// negate-A bit. This is the complex trailing update the BatchLAS pages list among
// their potrf types ("BatchLAS perf_blackwell", the cfloat potrf rows), here on
// tcgen05 with the accumulators in tensor memory.
//
// One block (256 threads) per output tile (I, K), I >= K, on a one-dimensional
// grid with the tile index fastest. The k dimension goes through shared memory
// 8 complex columns at a time in a ring of three buffers: threads 0..127 stage
// the I rows, 128..255 the K rows (a diagonal tile's two operands are the same
// rows, staged once); a thread loads two rows x four complex columns (16-byte
// loads, two complex numbers each, down the columns), splits real and imaginary
// parts into hi and lo and writes them K-major. Thread 0 issues the twelve MMAs
// of a slice, commits them to the buffer's mbarrier and alone waits, one slice
// ahead of the buffer's reuse. Every wait is bounded; a block that gives up marks
// the matrix info = -1, drains its MMAs and still releases its tensor memory.
#include <mutex>

#include "bl_common.cuh"
#include "launch.cuh"
#include "tc_sm100.cuh"

namespace bl {
namespace {

constexpr int kNb = 128;                         // panel width (complex columns)
constexpr int kKs = 8;                           // complex k per slice (one MMA k-step)
constexpr int kSlices = kNb / kKs;               // 16
constexpr uint32_t kLbo = 128;                   // K-adjacent core matrices
constexpr uint32_t kSbo = (kKs / 4) * 128 + 16;  // row-group stride, +16 B: no bank conflicts
constexpr uint32_t kTileBytes = 16 * kSbo;       // 128 rows x 8 k
constexpr uint32_t kOpBytes = 4 * kTileBytes;    // P hi, P lo, Q hi, Q lo of one operand
constexpr uint32_t kStageBytes = 2 * kOpBytes;   // the I and the K operand
constexpr int kStages = 3;
constexpr int kSmemBytes = kStages * kStageBytes;
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s at 2 GHz
constexpr uint32_t kNegateA = 1u << 13;          // instruction descriptor: negate A

// failure injection for the give-up test (see set_fail_first_wait in launch.cuh)
__device__ int g_fail_first_wait;

__device__ __forceinline__ uint32_t core_off(int r, int kq)
{
    // byte offset of (row r, k = 4kq .. 4kq+3) in a K-major no-swizzle tile
    return (uint32_t)(r >> 3) * kSbo + (uint32_t)kq * kLbo + (uint32_t)(r & 7) * 16;
}

template <bool UP>
__global__ void __launch_bounds__(256, 2)
cherk_tc_kernel(float2 *__restrict__ A, int n, int lda, int64_t strideA, int c0, int ntiles_col,
                int *__restrict__ info)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint32_t tmem_base;
    __shared__ __align__(8) uint64_t mbar[kStages];
    __shared__ int sh_err;

    const int nt = ntiles_col * (ntiles_col + 1) / 2;  // tiles a matrix
    const int64_t mat = blockIdx.x / nt;
    const int tile = (int)(blockIdx.x % nt);
    pdl_wait();
    pdl_trigger();
    if (block_skip(info, mat)) return;
    int I, K;
    {
        int i = (int)((sqrtf(8.0f * (float)tile + 1.0f) - 1.0f) * 0.5f);
        while ((i + 1) * (i + 2) / 2 <= tile) ++i;
        while (i * (i + 1) / 2 > tile) --i;
        I = i;
        K = tile - i * (i + 1) / 2;
    }
    float2 *__restrict__ Ab = A + mat * strideA;
    const int c1 = c0 + kNb;
    const int m = n - c1;
    const int ri = I * 128, rk = K * 128;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // staging: op 0 the I rows, op 1 the K rows; rows 2rp, 2rp + 1, complex
    // columns 4kq .. 4kq + 3 of the slice
    const int op = tid >> 7;
    const bool stager = !(op == 1 && I == K);
    const int rp = tid & 63, kq = (tid >> 6) & 1;
    const int rbase = op ? rk : ri;
    // lower storage: src[c lda] holds rows 2rp, 2rp + 1 of complex column c;
    // upper: row 2rp + i of the operand is the contiguous column
    // c1 + rbase + 2rp + i of U, src + i lda its columns 4kq ..
    const float2 *src = UP ? Ab + (c0 + 4 * kq) + (int64_t)(c1 + rbase + 2 * rp) * lda
                           : Ab + (c1 + rbase + 2 * rp) + (int64_t)(c0 + 4 * kq) * lda;
    const int valid_rows = max(0, min(2, m - rbase - 2 * rp));

    if (tid == 0) {
        sh_err = 0;
        for (int i = 0; i < kStages; ++i) tc::mbar_init(&mbar[i], 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, 256);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base;
    const uint32_t sbase = tc::smem_u32(smem);
    constexpr uint32_t idesc = tc::idesc_tf32(128, 128);

    // v[c]: complex column 4kq + c of rows 2rp, 2rp + 1: (re, im, re, im)
    float4 cur[4], nxt[4], nxt2[4];
    auto load_slice = [&](int s, float4 (&v)[4]) {
        if (!stager) return;
        if constexpr (UP) {
            // U's raw values: the conjugates of L's at the transposed places, so
            // the same products give the conjugate of the lower update, which is
            // what the upper triangle stores
            float4 r[2][2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float2 *p = src + (int64_t)i * lda + s * kKs;
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    r[i][h] = i < valid_rows ? *reinterpret_cast<const float4 *>(p + 2 * h)
                                             : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float4 a = r[0][c >> 1], b = r[1][c >> 1];
                v[c] = (c & 1) ? make_float4(a.z, a.w, b.z, b.w) : make_float4(a.x, a.y, b.x, b.y);
            }
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float2 *p = src + (int64_t)(s * kKs + c) * lda;
                if (valid_rows == 2) {
                    v[c] = *reinterpret_cast<const float4 *>(p);
                } else {
                    const float2 a = valid_rows > 0 ? p[0] : make_float2(0.0f, 0.0f);
                    v[c] = make_float4(a.x, a.y, 0.0f, 0.0f);
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
    for (int s = 0; s < kSlices; ++s) {
        // slice s goes to buffer s % 3, whose MMAs (slice s - 3) thread 0 saw
        // complete before the previous slice's barrier
        const int b = s % kStages;
        if (s + 2 < kSlices) load_slice(s + 2, nxt2);  // two slices in flight
        if (stager) {
            uint8_t *st = smem + b * kStageBytes + op * kOpBytes;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                float ph[4], pl[4], qh[4], ql[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    tc::split_tf32(i ? cur[c].z : cur[c].x, ph[c], pl[c]);
                    tc::split_tf32(i ? cur[c].w : cur[c].y, qh[c], ql[c]);
                }
                const uint32_t off = core_off(2 * rp + i, kq);
                *reinterpret_cast<float4 *>(st + off) = make_float4(ph[0], ph[1], ph[2], ph[3]);
                *reinterpret_cast<float4 *>(st + kTileBytes + off) =
                    make_float4(pl[0], pl[1], pl[2], pl[3]);
                *reinterpret_cast<float4 *>(st + 2 * kTileBytes + off) =
                    make_float4(qh[0], qh[1], qh[2], qh[3]);
                *reinterpret_cast<float4 *>(st + 3 * kTileBytes + off) =
                    make_float4(ql[0], ql[1], ql[2], ql[3]);
            }
        }
        tc::fence_async_smem();
        // thread 0 waits for the MMAs of slice s - 2 (the buffer the next slice
        // overwrites); the block barrier passes it on
        if (tid == 0 && s >= 2 &&
            ((s == 2 && fail_first) ||
             !tc::mbar_wait(&mbar[(s - 2) % kStages], ((s - 2) / kStages) & 1, kWaitCycles)))
            sh_err = 1;
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (sh_err) { ok = false; break; }
        if (tid == 0) {
            const uint32_t oi = sbase + b * kStageBytes;
            const uint32_t ok_ = I == K ? oi : oi + kOpBytes;
            const uint32_t pih = oi, pil = oi + kTileBytes, qih = oi + 2 * kTileBytes,
                           qil = oi + 3 * kTileBytes;
            const uint32_t pkh = ok_, pkl = ok_ + kTileBytes, qkh = ok_ + 2 * kTileBytes,
                           qkl = ok_ + 3 * kTileBytes;
            const uint32_t acc0 = s > 0 ? 1u : 0u;
            auto d = [](uint32_t a) { return tc::smem_desc(a, kLbo, kSbo); };
            // real part: P_I P_K^T + Q_I Q_K^T
            tc::mma_tf32(tmem, d(pih), d(pkh), idesc, acc0);
            tc::mma_tf32(tmem, d(pih), d(pkl), idesc, 1u);
            tc::mma_tf32(tmem, d(pil), d(pkh), idesc, 1u);
            tc::mma_tf32(tmem, d(qih), d(qkh), idesc, 1u);
            tc::mma_tf32(tmem, d(qih), d(qkl), idesc, 1u);
            tc::mma_tf32(tmem, d(qil), d(qkh), idesc, 1u);
            // imaginary part: Q_I P_K^T - P_I Q_K^T
            tc::mma_tf32(tmem + 128, d(qih), d(pkh), idesc, acc0);
            tc::mma_tf32(tmem + 128, d(qih), d(pkl), idesc, 1u);
            tc::mma_tf32(tmem + 128, d(qil), d(pkh), idesc, 1u);
            tc::mma_tf32(tmem + 128, d(pih), d(qkh), idesc | kNegateA, 1u);
            tc::mma_tf32(tmem + 128, d(pih), d(qkl), idesc | kNegateA, 1u);
            tc::mma_tf32(tmem + 128, d(pil), d(qkh), idesc | kNegateA, 1u);
            tc::mma_commit(&mbar[b]);
        }
        ++issued;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            cur[c] = nxt[c];
            nxt[c] = nxt2[c];
        }
    }

    const int last = issued - 1;
    if (tid == 0 && ok && !tc::mbar_wait(&mbar[last % kStages], (last / kStages) & 1, kWaitCycles))
        sh_err = 1;
    __syncthreads();
    ok = sh_err == 0;
    tc::fence_after_sync();

    // warp w: accumulator rows 32 (w % 4) .., columns 64 (w / 4) ..; the tile's
    // element (r, c) is complex entry (c1 + ri + r) + (c1 + rk + c) lda
    const int q = warp & 3, h = warp >> 2;
    const int r = 32 * q + lane;
    const int gr = ri + r;
    // element (r, c) of the tile: lower storage at (c1 + gr) + (c1 + gc) lda,
    // upper at (c1 + gc) + (c1 + gr) lda (a lane's 16 columns contiguous)
    float2 *Crow = UP ? Ab + c1 + (int64_t)(c1 + gr) * lda : Ab + (c1 + gr) + (int64_t)c1 * lda;
    const int64_t cs = UP ? 1 : lda;
    if (ok) {
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
            const int gc0 = rk + 64 * h + 16 * cc;
            float2 old[16];
            if constexpr (UP) {
                // a lane's 16 entries are contiguous: 16-byte accesses by pairs,
                // a single entry where only the first of a pair is in the triangle
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    const int gc = gc0 + j;
                    const bool in0 = gr < m && gc < m && gr >= gc;
                    const bool in1 = gr < m && gc + 1 < m && gr >= gc + 1;
                    if (in1) {
                        const float4 o = *reinterpret_cast<const float4 *>(Crow + gc);
                        old[j] = make_float2(o.x, o.y);
                        old[j + 1] = make_float2(o.z, o.w);
                    } else {
                        old[j] = in0 ? Crow[gc] : make_float2(0.0f, 0.0f);
                        old[j + 1] = make_float2(0.0f, 0.0f);
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int gc = gc0 + j;
                    old[j] = (gr < m && gc < m && gr >= gc) ? Crow[(int64_t)gc * cs]
                                                           : make_float2(0.0f, 0.0f);
                }
            }
            float vr[16], vi[16];
            tc::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + 64 * h + 16 * cc, vr);
            tc::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + 128 + 64 * h + 16 * cc, vi);
            if constexpr (UP) {
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    const int gc = gc0 + j;
                    const bool in0 = gr < m && gc < m && gr >= gc;
                    const bool in1 = gr < m && gc + 1 < m && gr >= gc + 1;
                    if (in1)
                        *reinterpret_cast<float4 *>(Crow + gc) =
                            make_float4(old[j].x - vr[j], old[j].y - vi[j], old[j + 1].x - vr[j + 1],
                                        old[j + 1].y - vi[j + 1]);
                    else if (in0)
                        Crow[gc] = make_float2(old[j].x - vr[j], old[j].y - vi[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int gc = gc0 + j;
                    if (gr < m && gc < m && gr >= gc)
                        Crow[(int64_t)gc * cs] = make_float2(old[j].x - vr[j], old[j].y - vi[j]);
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
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// Returns 0 after launching, 1 when the complex panels are not 16-byte aligned
// (the caller's FP32 kernel), -1 on a trailing matrix that is empty.
template <bool UP>
int launch_t(float *A, int n, int lda, int64_t strideA, int batch, int *info, int c0,
             cudaStream_t stream)
{
    if (((reinterpret_cast<uintptr_t>(A) & 15) != 0) || (lda & 1) || (strideA & 1)) return 1;
    const int m = n - c0 - kNb;
    if (m <= 0) return -1;
    static DeviceOnce attrs;
    if (const int e = attrs.run([] {
            return cudaFuncSetAttribute(cherk_tc_kernel<UP>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        }))
        return e;
    const int T = (m + 127) / 128;
    const int64_t blocks = (int64_t)batch * (T * (T + 1) / 2);
    if (blocks > 0x7fffffffLL) return (int)cudaErrorInvalidConfiguration;
    return launch_pdl(cherk_tc_kernel<UP>, dim3((unsigned)blocks), dim3(256), (size_t)kSmemBytes,
                      stream, reinterpret_cast<float2 *>(A), n, lda, strideA, c0, T, info);
}

}  // namespace

int set_fail_first_wait_cherk_tc(int every)
{
    return (int)cudaMemcpyToSymbol(g_fail_first_wait, &every, sizeof every);
}

int launch_cherk_tc(float *A, int n, int lda, int64_t strideA, int batch, int *info, int c0,
                    cudaStream_t stream, bool upper)
{
    return upper ? launch_t<true>(A, n, lda, strideA, batch, info, c0, stream)
                 : launch_t<false>(A, n, lda, strideA, batch, info, c0, stream);
}

}  // namespace bl
