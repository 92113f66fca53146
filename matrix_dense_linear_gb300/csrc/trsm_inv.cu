// Panel solve of the blocked path by the inverse of the diagonal block:
//     W   = L11^{-1}                      (one block per matrix, FP32)
//     L21 = A21 L11^{-T} = A21 W^T        (one 3xTF32 tensor-core GEMM tile per 128 rows)
// instead of the forward substitution of trsm_tc.cu. This is the panel solve
// of "kernelbot-cholesky-930185" (changelog sections "THE MECHANISM, FOR THE
// NEXT BUILD" and "WHY tri_inv IS SHAPED THE WAY IT IS": a triangular solve
// cannot use the tensor cores, a multiply by the inverse can; the inverse is
// computed with one thread per column, the column recurrence reading only L
// and that column's earlier entries). The inverse is computed once per matrix
// and panel and shared by every row block of the panel through the caller's
// workspace W (128 x 128 floats per matrix, row-major: W[c * 128 + k] =
// (L11^{-1})(c, k), zero above the diagonal), so it pays where a panel has
// many rows below its diagonal block (large n).
//
// Multiplying by an explicit inverse is less stable than substitution: the
// error of L21 grows with the condition of L11 (its square root of A11's),
// which the parity tests bound on the workloads' spectra.
#include <mutex>

#include "bl_common.cuh"
#include "launch.cuh"
#include "tc_sm100.cuh"

namespace bl {
namespace {

constexpr int kNb = 128;
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s at 2 GHz

// L11 in shared memory packed by 32-column blocks: block b keeps rows
// 32b .. 127 of its 32 columns, column-major with leading dimension 128 - 32b.
__host__ __device__ constexpr int l11_off(int b) { return 32 * (128 * b - 32 * (b * (b - 1) / 2)); }
constexpr int kL11Floats = l11_off(4);  // 10240 floats, 40 KB
__device__ __forceinline__ const float *l11_col(const float *Ls, int k)
{
    // pointer p with p[i] = L11(i, k) for i >= 32*(k/32)
    const int b = k >> 5;
    return Ls + l11_off(b) + (k - 32 * b) * (128 - 32 * b) - 32 * b;
}
constexpr int kInvSmem = (kL11Floats + kNb * kNb) * 4;  // packed L11 + X, 104 KB

// W = L11^{-1}. Thread c computes column c of the inverse, x = L11^{-1} e_c,
// by row blocks R of 32: the right-hand side of block R is e_c minus the
// contributions L(R, R') x(R') of the finished blocks R' < R (read back from
// the inverse in shared memory, the thread's own column), then a forward
// substitution against the diagonal block L(R, R) with its reciprocal
// diagonal. A warp's 32 columns are zero above row 32 * warp, so its earlier
// row blocks are skipped (uniformly).
template <bool UP>
__global__ void __launch_bounds__(128, 2)
trinv_kernel(const float *__restrict__ A, int n, int lda, int64_t strideA, int c0,
             float *__restrict__ W, int *__restrict__ info)
{
    extern __shared__ __align__(16) float sm[];
    float *Ls = sm;                  // packed L11
    float *X = sm + kL11Floats;      // X[row * 128 + col] = inverse(row, col)
    __shared__ float rinv[kNb];
    const int64_t mat = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    if (block_skip(info, mat)) return;
    const float *L11 = A + mat * strideA + c0 + (int64_t)c0 * lda;  // (c0, c0), either storage
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int j = warp; j < kNb; j += 4) {
        float *dst = const_cast<float *>(l11_col(Ls, j));
        for (int i = j + lane; i < kNb; i += 32) cp_async4(dst + i, L11 + lidx<UP>(i, j, lda));
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    rinv[tid] = 1.0f / l11_col(Ls, tid)[tid];
    __syncthreads();

    const int c = tid;
#pragma unroll 1
    for (int R = 0; R < 4; ++R) {
        float b[32];
        if (R < warp) {  // rows above this warp's columns: zero
#pragma unroll
            for (int i = 0; i < 32; ++i) X[(32 * R + i) * kNb + c] = 0.0f;
            continue;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) b[i] = (32 * R + i == c) ? 1.0f : 0.0f;
#pragma unroll 1
        for (int Rp = warp; Rp < R; ++Rp) {
#pragma unroll 4
            for (int t = 0; t < 32; ++t) {
                const float xk = X[(32 * Rp + t) * kNb + c];
                const float4 *Lc = reinterpret_cast<const float4 *>(l11_col(Ls, 32 * Rp + t) + 32 * R);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 l4 = Lc[q];
                    b[4 * q + 0] = fmaf(-l4.x, xk, b[4 * q + 0]);
                    b[4 * q + 1] = fmaf(-l4.y, xk, b[4 * q + 1]);
                    b[4 * q + 2] = fmaf(-l4.z, xk, b[4 * q + 2]);
                    b[4 * q + 3] = fmaf(-l4.w, xk, b[4 * q + 3]);
                }
            }
        }
        // the diagonal block: Ld[i + t * ld] = L11(32R + i, 32R + t)
        const float *Ld = l11_col(Ls, 32 * R) + 32 * R;
        const int ld = kNb - 32 * R;
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            b[t] *= rinv[32 * R + t];
#pragma unroll
            for (int q = (t + 1) / 4; q < 8; ++q) {
                const float4 l4 = reinterpret_cast<const float4 *>(Ld + t * ld)[q];
                const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = 4 * q + u;
                    if (i > t) b[i] = fmaf(-lv[u], b[t], b[i]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) X[(32 * R + i) * kNb + c] = b[i];
    }
    __syncthreads();
    float4 *Wm = reinterpret_cast<float4 *>(W + mat * (int64_t)(kNb * kNb));
    const float4 *Xs = reinterpret_cast<const float4 *>(X);
#pragma unroll 4
    for (int e = tid; e < kNb * kNb / 4; e += 128) Wm[e] = Xs[e];
}

// ---------------------------------------------------------------------------
// L21 = A21 W^T: one block (256 threads) per 128 rows below the diagonal
// block. Operand P = those rows of A21 (k = the panel's 128 columns), operand
// Q = W (row c of W = row c of the inverse); the k dimension goes through
// shared memory 16 columns at a time (a ring of three buffers), each operand split into
// a TF32-exact high part and the FP32 remainder and written K-major (threads
// 0..127 stage P, 128..255 stage Q; 16-byte loads down the columns of P in
// the lower storage, along the rows otherwise), and thread 0 issues three
// tcgen05.mma of M = N = 128, K = 8 per k-step (hi hi, hi lo, lo hi) into one
// tensor-memory accumulator. The epilogue stores the accumulator over A21
// (every row of the block was read before the first store). The lower
// storage computes D = P Q^T (lane = row, the rows of a column contiguous in
// memory); the upper one D = Q P^T (lane = column, a row contiguous).
// ---------------------------------------------------------------------------
constexpr int kKs = 16;                    // k columns per shared-memory slice
constexpr int kSlices = kNb / kKs;         // 8
constexpr uint32_t kLbo = 128;             // K-adjacent core matrices
constexpr uint32_t kSbo = (kKs / 4) * 128 + 16;  // row-group stride, +16 B: no bank conflicts
constexpr uint32_t kTileBytes = 16 * kSbo;  // 128 rows
constexpr uint32_t kStageBytes = 4 * kTileBytes;  // P hi, P lo, Q hi, Q lo
constexpr int kStages = 3;                 // operand buffers in the ring
constexpr int kGemmSmem = kStages * kStageBytes;

// failure injection for the give-up test (see set_fail_first_wait in launch.cuh)
__device__ int g_fail_first_wait;

__device__ __forceinline__ uint32_t core_off(int r, int kq)
{
    // byte offset of (row r, k = 4kq .. 4kq+3) in a K-major no-swizzle tile
    return (uint32_t)(r >> 3) * kSbo + (uint32_t)kq * kLbo + (uint32_t)(r & 7) * 16;
}

template <bool UP>
__global__ void __launch_bounds__(256, 2)
trsm_gemm_kernel(float *__restrict__ A, int n, int lda, int64_t strideA, int c0, int nrb,
                 const float *__restrict__ W, int *__restrict__ info)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint32_t tmem_base;
    __shared__ __align__(8) uint64_t mbar[kStages];
    __shared__ int sh_err;

    // one-dimensional grid, the row block fastest: a matrix's row blocks run
    // together and read its inverse from L2
    const int64_t mat = blockIdx.x / nrb;
    const int rb = (int)(blockIdx.x % nrb);
    pdl_wait();
    pdl_trigger();
    if (block_skip(info, mat)) return;
    float *__restrict__ Ab = A + mat * strideA;
    const float *Wm = W + mat * (int64_t)(kNb * kNb);
    const int R0 = c0 + kNb + kNb * rb;  // first row of this block
    const int rows = n - R0 < kNb ? n - R0 : kNb;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // staging: op 0 the rows of A21 (P), op 1 the inverse (Q); kc: the operand's
    // rows are contiguous along k in memory (16-byte loads along a row, 4 rows
    // a thread), else 16-byte loads down 4 columns
    const int op = tid >> 7;
    const bool kc = op == 1 || UP;
    const int rq = kc ? (tid >> 2) & 31 : tid & 31;  // row quad: rows 4rq .. 4rq+3
    const int kq = kc ? tid & 3 : (tid >> 5) & 3;    // k quad within the slice
    const float *src = op ? Wm + 4 * rq * kNb + 4 * kq : Ab + lidx<UP>(R0 + 4 * rq, c0 + 4 * kq, lda);
    const int64_t rstep = op ? kNb : lda;  // between consecutive rows (kc) or k columns (!kc)
    const int valid_rows = op ? 4 : max(0, min(4, rows - 4 * rq));

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

    // kc: v[i] = row 4rq + i, k = 4kq .. 4kq+3; else v[c] = k = 4kq + c, rows 4rq .. 4rq+3
    float4 cur[4], nxt[4], nxt2[4];
    auto load_slice = [&](int s, float4 (&v)[4]) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (kc) {
                const float *p = src + (int64_t)c * rstep + s * kKs;
                v[c] = valid_rows > c ? *reinterpret_cast<const float4 *>(p)
                                      : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            } else {
                const float *p = src + (int64_t)(s * kKs + c) * rstep;
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
    for (int s = 0; s < kSlices; ++s) {
        // a three-buffer ring: slice s goes to buffer s % 3, whose MMAs (slice
        // s - 3) thread 0 saw complete before the previous slice's barrier
        const int b = s % kStages;
        if (s + 2 < kSlices) load_slice(s + 2, nxt2);  // two slices in flight
        uint8_t *st = smem + b * kStageBytes + (op ? 2 : 0) * kTileBytes;
        const float cv[4][4] = {{cur[0].x, cur[0].y, cur[0].z, cur[0].w},
                                {cur[1].x, cur[1].y, cur[1].z, cur[1].w},
                                {cur[2].x, cur[2].y, cur[2].z, cur[2].w},
                                {cur[3].x, cur[3].y, cur[3].z, cur[3].w}};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float h[4], l[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) tc::split_tf32(kc ? cv[i][c] : cv[c][i], h[c], l[c]);
            const uint32_t off = core_off(4 * rq + i, kq);
            *reinterpret_cast<float4 *>(st + off) = make_float4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<float4 *>(st + kTileBytes + off) = make_float4(l[0], l[1], l[2], l[3]);
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
            const uint32_t p_hi = sbase + b * kStageBytes, p_lo = p_hi + kTileBytes;
            const uint32_t q_hi = p_hi + 2 * kTileBytes, q_lo = p_hi + 3 * kTileBytes;
#pragma unroll
            for (int ks = 0; ks < kKs / 8; ++ks) {
                const uint32_t ko = ks * 2 * kLbo;
                const uint32_t acc0 = (s > 0 || ks > 0) ? 1u : 0u;
                // (hi_P, hi_Q), (hi_P, lo_Q), (lo_P, hi_Q) in both storages; the
                // upper storage swaps the MMA operands (D = Q P^T)
                const uint32_t a0 = UP ? q_hi : p_hi, b0 = UP ? p_hi : q_hi;
                const uint32_t a1 = UP ? q_lo : p_hi, b1 = UP ? p_hi : q_lo;
                const uint32_t a2 = UP ? q_hi : p_lo, b2 = UP ? p_lo : q_hi;
                tc::mma_tf32(tmem, tc::smem_desc(a0 + ko, kLbo, kSbo),
                             tc::smem_desc(b0 + ko, kLbo, kSbo), idesc, acc0);
                tc::mma_tf32(tmem, tc::smem_desc(a1 + ko, kLbo, kSbo),
                             tc::smem_desc(b1 + ko, kLbo, kSbo), idesc, 1u);
                tc::mma_tf32(tmem, tc::smem_desc(a2 + ko, kLbo, kSbo),
                             tc::smem_desc(b2 + ko, kLbo, kSbo), idesc, 1u);
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

    const int last = issued - 1;
    if (tid == 0 && ok && !tc::mbar_wait(&mbar[last % kStages], (last / kStages) & 1, kWaitCycles))
        sh_err = 1;
    __syncthreads();
    ok = sh_err == 0;
    tc::fence_after_sync();

    // warp w: accumulator lanes 32 (w % 4) .., columns 64 (w / 4) ..
    const int q = warp & 3, h = warp >> 2;
    const int dl = 32 * q + lane;  // this thread's accumulator row
    if (ok) {
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
            float v[16];
            tc::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + 64 * h + 16 * cc, v);
            if constexpr (UP) {
                // lower-storage view: D(c, r) = L21(R0 + r, c0 + c), c = dl
                float *out = Ab + (c0 + dl) + (int64_t)R0 * lda;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int r = 64 * h + 16 * cc + j;
                    if (r < rows) out[(int64_t)r * lda] = v[j];
                }
            } else {
                // D(r, c) = L21(R0 + r, c0 + c), r = dl
                float *out = Ab + (R0 + dl) + (int64_t)c0 * lda;
                if (dl < rows) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        out[(int64_t)(64 * h + 16 * cc + j) * lda] = v[j];
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
int launch_u(float *A, int n, int lda, int64_t strideA, int batch, int *info, int c0, float *W,
             cudaStream_t stream)
{
    static DeviceOnce attrs;
    if (const int e = attrs.run([] {
            int e1 = (int)cudaFuncSetAttribute(trinv_kernel<UP>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kInvSmem);
            if (e1) return (cudaError_t)e1;
            return cudaFuncSetAttribute(trsm_gemm_kernel<UP>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
        }))
        return e;
    int e = launch_pdl(trinv_kernel<UP>, dim3((unsigned)batch), dim3(128), (size_t)kInvSmem,
                       stream, (const float *)A, n, lda, strideA, c0, W, info);
    if (e) return e;
    const int m = n - c0 - kNb;
    const int nrb = (m + kNb - 1) / kNb;
    const int64_t blocks = (int64_t)batch * nrb;
    if (blocks > 0x7fffffffLL) return (int)cudaErrorInvalidConfiguration;
    return launch_pdl(trsm_gemm_kernel<UP>, dim3((unsigned)blocks), dim3(256),
                      (size_t)kGemmSmem, stream, A, n, lda, strideA, c0, nrb, (const float *)W,
                      info);
}

}  // namespace

int set_fail_first_wait_trsm_inv(int every)
{
    return (int)cudaMemcpyToSymbol(g_fail_first_wait, &every, sizeof every);
}

int launch_trsm_inv(float *A, int n, int lda, int64_t strideA, int batch, int *info, int c0,
                    float *W, cudaStream_t stream, bool upper)
{
    if (((reinterpret_cast<uintptr_t>(A) & 15) != 0) || (lda & 3) || (strideA & 3) ||
        ((reinterpret_cast<uintptr_t>(W) & 15) != 0))
        return 1;
    if (n - c0 - kNb <= 0) return -1;
    return upper ? launch_u<true>(A, n, lda, strideA, batch, info, c0, W, stream)
                 : launch_u<false>(A, n, lda, strideA, batch, info, c0, W, stream);
}

}  // namespace bl
