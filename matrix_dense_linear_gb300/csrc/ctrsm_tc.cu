// Panel solve of the single-precision complex blocked path with the tensor
// cores doing the block updates (either storage; the upper one reads and writes
// U = L^H's raw values at the transposed places, the conjugates of L's, so the
// same arithmetic yields the conjugated results it stores):
//     L21 = A21 L11^{-H}      (A21: the rows below the 128 x 128 diagonal block)
// as a blocked forward substitution over four 32-column blocks j:
//     X_j = (A_j - sum_{i<j} X_i L_ji^H) L_jj^{-H}.
// One block of 128 threads takes 128 rows, a thread a row. Tensor memory holds
// -(A21 rows) as two real halves, the real parts in columns 0..127 and the
// imaginary parts in 128..255 (lane = row). For j = 0..3 every thread reads its
// row's 32 complex columns of block j back and substitutes them against the
// diagonal block L_jj (real reciprocal diagonal; x_c conj(l) as four FMAs on
// the FP32 pipes). The finished X_j goes to memory and, split into its real and
// imaginary parts, each in the error-compensated 3xTF32 form (x = hi + lo, hi
// exact in TF32: hi hi + hi lo + lo hi), becomes the A operand of one group of
// tcgen05.mma that adds X_j L_{k,j}^H to every later column block k > j:
//     Re += Xr Lr^T + Xi Li^T,    Im += Xi Lr^T - Xr Li^T
// (the subtracted product through the instruction's negate-A bit), twelve MMAs
// a k-step of eight. Three quarters of the complex flops run on the tensor
// cores; this is the complex panel solve the BatchLAS pages list among their
// potrf types ("BatchLAS perf_blackwell", the cfloat potrf rows) with the
// accumulators in tensor memory.
//
// Shared memory (115 KB: two blocks share an SM): the X operand (four 16 KB
// tiles: real hi, real lo, imaginary hi, imaginary lo, K-major, no padding: a
// quarter warp writes eight consecutive rows of one core matrix), which also
// holds the current diagonal block L_jj while the row is solved; and the
// off-diagonal rows of one column block of L11 (four tiles, 96 rows at most),
// fetched into registers while the previous block is solved. Needs 16-byte
// aligned complex panels (the caller keeps the FP32 kernel otherwise). Every
// wait is bounded; a block that gives up marks info = -1, lets its MMAs drain
// and still releases its tensor memory.
#include <mutex>

#include "bl_common.cuh"
#include "launch.cuh"
#include "tc_sm100.cuh"

namespace bl {
namespace {

constexpr uint32_t kLbo = 128;                 // K-adjacent core matrices
constexpr uint32_t kSbo = 8 * 128;             // row groups (K = 32 a row)
constexpr uint32_t kXTile = 16 * kSbo;         // 128 rows x 32 k
constexpr uint32_t kOffX = 0;                  // Xr hi, Xr lo, Xi hi, Xi lo
constexpr uint32_t kOffLt = 4 * kXTile;        // Lr hi, Lr lo, Li hi, Li lo
constexpr uint32_t kLtMax = 4 * 12 * kSbo;     // 96 rows
constexpr uint32_t kOffRinv = kOffLt + kLtMax;
constexpr int kSmemBytes = (int)(kOffRinv + 128 * 4);
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s at 2 GHz
constexpr uint32_t kNegateA = 1u << 13;          // instruction descriptor: negate A

// failure injection for the give-up test (see set_fail_first_wait in launch.cuh)
__device__ int g_fail_first_wait;

__device__ __forceinline__ uint32_t core_off(int r, int kq)
{
    return (uint32_t)(r >> 3) * kSbo + (uint32_t)kq * kLbo + (uint32_t)(r & 7) * 16;
}

// rows of L_{k,j}, k > j, for column block j
__host__ __device__ constexpr int lt_rows(int j) { return 96 - 32 * j; }

// Column block j of L11 below its diagonal block in pieces of two rows
// (32(j+1) + 2p, + 1) by four complex columns (32j + 4kq ..): piece
// b = s + 2 (p + np h) has kq = 2h + s, so that a quarter warp's eight pieces
// cover one row group in two column quads. A thread owns pieces tid,
// tid + 128, tid + 256; load() fetches them (16-byte loads: two complex rows of
// a column), stage() writes the four operand tiles, the two rows of a piece in
// the order that puts a quarter warp's stores on eight distinct rows.
template <bool UP>
struct LtPieces {
    float4 v[3][4];  // [piece][column]: (re, im) of the two rows
    __device__ __forceinline__ void load(const float2 *L11, int lda, int j, int tid)
    {
        const int np = lt_rows(j) / 2;
#pragma unroll
        for (int u = 0; u < 3; ++u) {
            const int b = tid + 128 * u;
            if (b < 8 * np) {
                const int s = b & 1, p = (b >> 1) % np, h = (b >> 1) / np;
                const int r0 = 32 * (j + 1) + 2 * p, k0 = 32 * j + 4 * (2 * h + s);
                if constexpr (UP) {
                    // row r of the piece is U's contiguous column r: two 16-byte
                    // loads a row, regrouped by column
                    float4 w[2][2];
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const float2 *src = L11 + k0 + (int64_t)(r0 + i) * lda;
                        w[i][0] = *reinterpret_cast<const float4 *>(src);
                        w[i][1] = *reinterpret_cast<const float4 *>(src + 2);
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float4 a = w[0][c >> 1], bb = w[1][c >> 1];
                        v[u][c] = (c & 1) ? make_float4(a.z, a.w, bb.z, bb.w)
                                          : make_float4(a.x, a.y, bb.x, bb.y);
                    }
                } else {
                    const float2 *src = L11 + r0 + (int64_t)k0 * lda;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        v[u][c] = *reinterpret_cast<const float4 *>(src + (int64_t)c * lda);
                }
            }
        }
    }
    __device__ __forceinline__ void stage(uint8_t *lt, int j, int tid) const
    {
        const int np = lt_rows(j) / 2;
        const uint32_t T = (uint32_t)lt_rows(j) / 8 * kSbo;
#pragma unroll
        for (int u = 0; u < 3; ++u) {
            const int b = tid + 128 * u;
            if (b < 8 * np) {
                const int s = b & 1, p = (b >> 1) % np, h = (b >> 1) / np;
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const int i = s ^ w;
                    float rh[4], rl[4], ih[4], il[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        tc::split_tf32(i ? v[u][c].z : v[u][c].x, rh[c], rl[c]);
                        tc::split_tf32(i ? v[u][c].w : v[u][c].y, ih[c], il[c]);
                    }
                    const uint32_t off = core_off(2 * p + i, 2 * h + s);
                    *reinterpret_cast<float4 *>(lt + off) = make_float4(rh[0], rh[1], rh[2], rh[3]);
                    *reinterpret_cast<float4 *>(lt + T + off) = make_float4(rl[0], rl[1], rl[2], rl[3]);
                    *reinterpret_cast<float4 *>(lt + 2 * T + off) =
                        make_float4(ih[0], ih[1], ih[2], ih[3]);
                    *reinterpret_cast<float4 *>(lt + 3 * T + off) =
                        make_float4(il[0], il[1], il[2], il[3]);
                }
            }
        }
    }
};

// The diagonal block L_jj, lower part: thread tid fetches entries
// e = tid + 128u, (row k, column t) = (e & 31, e >> 5), into registers; put()
// writes them as Ld[32 t + k] (complex), columns contiguous.
template <bool UP>
struct LdPart {
    float2 v[8];
    __device__ __forceinline__ void load(const float2 *L11, int lda, int j, int tid)
    {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = tid + 128 * u, k = e & 31, t = e >> 5;
            const int64_t o = UP ? (32 * j + t) + (int64_t)(32 * j + k) * lda
                                 : (32 * j + k) + (int64_t)(32 * j + t) * lda;
            v[u] = k >= t ? L11[o] : make_float2(0.0f, 0.0f);
        }
    }
    __device__ __forceinline__ void put(float2 *Ld, int tid) const
    {
#pragma unroll
        for (int u = 0; u < 8; ++u) Ld[tid + 128 * u] = v[u];
    }
};

template <bool UP>
__global__ void __launch_bounds__(128, 2)
ctrsm_tc_kernel(float2 *__restrict__ A, int n, int lda, int64_t strideA, int c0, int nrb,
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
    pdl_wait();
    pdl_trigger();
    if (block_skip(info, mat)) return;
    float2 *__restrict__ Ab = A + mat * strideA;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int R = c0 + 128 + rb * 128 + tid;  // this thread's row
    const bool live = R < n;
    // L11(i, k) = L11[i + k lda]; in the upper storage U's raw value at the
    // transposed place, L11[k + i lda]: the conjugates of L's values, so that
    // the same arithmetic gives the conjugated results the upper triangle keeps
    const float2 *L11 = Ab + c0 + (int64_t)c0 * lda;
    float2 *Ld = reinterpret_cast<float2 *>(smem + kOffX);
    float *rinv = reinterpret_cast<float *>(smem + kOffRinv);
    uint8_t *Lt = smem + kOffLt;

    if (tid == 0) {
        sh_err = 0;
        tc::mbar_init(&mbar, 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, 256);
        tc::tmem_relinquish();
    }

    // the first column block's off-diagonal rows, its diagonal block and the
    // reciprocal diagonal travel with the first half of the row
    LtPieces<UP> pc;
    pc.load(L11, lda, 0, tid);
    LdPart<UP> dg;
    dg.load(L11, lda, 0, tid);
    const float dii = L11[tid + (int64_t)tid * lda].x;
    // element (R, c0 + c): g[c lda] (lower), g[c] (upper: U's column R)
    const float2 *g = Ab + (live ? (UP ? c0 + (int64_t)R * lda : R + (int64_t)c0 * lda) : 0);
    auto load_chunk = [&](int q, float (&re)[32], float (&im)[32]) {
        if constexpr (UP) {
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
                const float4 a = live ? *reinterpret_cast<const float4 *>(g + 32 * q + c)
                                      : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                re[c] = -a.x; im[c] = -a.y; re[c + 1] = -a.z; im[c + 1] = -a.w;
            }
        } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float2 a = live ? g[(int64_t)(32 * q + c) * lda] : make_float2(0.0f, 0.0f);
                re[c] = -a.x;
                im[c] = -a.y;
            }
        }
    };
    float xr[32], xi[32];
    load_chunk(0, xr, xi);
    pc.stage(Lt, 0, tid);
    dg.put(Ld, tid);
    rinv[tid] = 1.0f / dii;

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base;
    const uint32_t tlane = tmem + ((uint32_t)(32 * warp) << 16);
    tc::tmem_st32(tlane, xr);
    tc::tmem_st32(tlane + 128, xi);
#pragma unroll 1
    for (int q = 1; q < 4; ++q) {
        load_chunk(q, xr, xi);
        tc::tmem_st32(tlane + 32 * q, xr);
        tc::tmem_st32(tlane + 128 + 32 * q, xi);
    }

    const uint32_t sbase = tc::smem_u32(smem);
    // the MMA group committed last and not yet seen complete (thread 0; -1: none)
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
            // the operand tiles are free again: block j's diagonal block and
            // off-diagonal rows
            dg.put(Ld, tid);
            if (j < 3) pc.stage(Lt, j, tid);
            __syncthreads();
        }
        // block j+1's pieces of L11 travel while block j is solved
        if (j + 1 < 3) pc.load(L11, lda, j + 1, tid);
        if (j + 1 < 4) dg.load(L11, lda, j + 1, tid);
        tc::tmem_ld32(tlane + 32 * j, xr);
        tc::tmem_ld32(tlane + 128 + 32 * j, xi);
        const float4 *Ld4 = reinterpret_cast<const float4 *>(Ld);
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            const float rt = rinv[32 * j + t];
            xr[t] = -xr[t] * rt;
            xi[t] = -xi[t] * rt;
#pragma unroll
            for (int q = (t + 1) / 2; q < 16; ++q) {
                const float4 l2 = Ld4[t * 16 + q];  // L(2q, t), L(2q + 1, t) of the block
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int k = 2 * q + u;
                    if (k > t) {  // y_k += x_t conj(l_kt)
                        const float lr = u ? l2.z : l2.x, li = u ? l2.w : l2.y;
                        xr[k] = fmaf(xr[t], lr, fmaf(xi[t], li, xr[k]));
                        xi[k] = fmaf(xi[t], lr, fmaf(-xr[t], li, xi[k]));
                    }
                }
            }
        }
        if (live) {
            if constexpr (UP) {
                float2 *out = Ab + (c0 + 32 * j) + (int64_t)R * lda;
#pragma unroll
                for (int t = 0; t < 32; t += 2)
                    *reinterpret_cast<float4 *>(out + t) = make_float4(xr[t], xi[t], xr[t + 1], xi[t + 1]);
            } else {
                float2 *out = Ab + R + (int64_t)(c0 + 32 * j) * lda;
#pragma unroll
                for (int t = 0; t < 32; ++t) out[(int64_t)t * lda] = make_float2(xr[t], xi[t]);
            }
        }
        if (j == 3) break;
        __syncthreads();  // every thread is done with Ld before X overwrites it
        // X_j as the A operand (K-major, hi/lo of the real and imaginary parts)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float rh[4], rl[4], ih[4], il[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                tc::split_tf32(xr[4 * q + u], rh[u], rl[u]);
                tc::split_tf32(xi[4 * q + u], ih[u], il[u]);
            }
            const uint32_t off = core_off(tid, q);
            uint8_t *x = smem + kOffX;
            *reinterpret_cast<float4 *>(x + off) = make_float4(rh[0], rh[1], rh[2], rh[3]);
            *reinterpret_cast<float4 *>(x + kXTile + off) = make_float4(rl[0], rl[1], rl[2], rl[3]);
            *reinterpret_cast<float4 *>(x + 2 * kXTile + off) = make_float4(ih[0], ih[1], ih[2], ih[3]);
            *reinterpret_cast<float4 *>(x + 3 * kXTile + off) = make_float4(il[0], il[1], il[2], il[3]);
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (tid == 0) {
            // -A[:, 32(j+1):] += X_j L_{k,j}^H   (M = 128, N = 96 - 32j, K = 32)
            const uint32_t N = (uint32_t)lt_rows(j);
            const uint32_t T = N / 8 * kSbo;
            const uint32_t idesc = tc::idesc_tf32(128, N);
            const uint32_t drd = tmem + 32 * (j + 1), did = drd + 128;
            auto d = [](uint32_t a) { return tc::smem_desc(a, kLbo, kSbo); };
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint32_t ko = ks * 2 * kLbo;
                const uint32_t xrh = sbase + kOffX + ko, xrl = xrh + kXTile, xih = xrh + 2 * kXTile,
                               xil = xrh + 3 * kXTile;
                const uint32_t lrh = sbase + kOffLt + ko, lrl = lrh + T, lih = lrh + 2 * T,
                               lil = lrh + 3 * T;
                // real part: Xr Lr^T + Xi Li^T
                tc::mma_tf32(drd, d(xrh), d(lrh), idesc, 1u);
                tc::mma_tf32(drd, d(xrh), d(lrl), idesc, 1u);
                tc::mma_tf32(drd, d(xrl), d(lrh), idesc, 1u);
                tc::mma_tf32(drd, d(xih), d(lih), idesc, 1u);
                tc::mma_tf32(drd, d(xih), d(lil), idesc, 1u);
                tc::mma_tf32(drd, d(xil), d(lih), idesc, 1u);
                // imaginary part: Xi Lr^T - Xr Li^T
                tc::mma_tf32(did, d(xih), d(lrh), idesc, 1u);
                tc::mma_tf32(did, d(xih), d(lrl), idesc, 1u);
                tc::mma_tf32(did, d(xil), d(lrh), idesc, 1u);
                tc::mma_tf32(did, d(xrh), d(lih), idesc | kNegateA, 1u);
                tc::mma_tf32(did, d(xrh), d(lil), idesc | kNegateA, 1u);
                tc::mma_tf32(did, d(xrl), d(lih), idesc | kNegateA, 1u);
            }
            tc::mma_commit(&mbar);
            pend = j;
        }
    }

    // a block that gave up lets its last MMA group drain (bounded) first: no
    // MMA may still write the tensor memory it releases
    if (tid == 0 && sh_err && pend >= 0) tc::mbar_wait(&mbar, pend & 1, kWaitCycles);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
    if (tid == 0 && sh_err) info[mat] = -1;
}

template <bool UP>
int launch_t(float *A, int n, int lda, int64_t strideA, int batch, int *info, int c0,
             cudaStream_t stream)
{
    if (((reinterpret_cast<uintptr_t>(A) & 15) != 0) || (lda & 1) || (strideA & 1)) return 1;
    const int m = n - c0 - 128;
    if (m <= 0) return -1;
    static DeviceOnce attrs;
    if (const int e = attrs.run([] {
            return cudaFuncSetAttribute(ctrsm_tc_kernel<UP>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        }))
        return e;
    const int nrb = (m + 127) / 128;
    const int64_t blocks = (int64_t)batch * nrb;
    if (blocks > 0x7fffffffLL) return (int)cudaErrorInvalidConfiguration;
    return launch_pdl(ctrsm_tc_kernel<UP>, dim3((unsigned)blocks), dim3(128), (size_t)kSmemBytes,
                      stream, reinterpret_cast<float2 *>(A), n, lda, strideA, c0, nrb, info);
}

}  // namespace

int set_fail_first_wait_ctrsm_tc(int every)
{
    return (int)cudaMemcpyToSymbol(g_fail_first_wait, &every, sizeof every);
}

// Returns 0 after launching, 1 when the complex panels are not 16-byte aligned
// (the caller's FP32 kernel), -1 on an empty panel, or a cudaError_t.
int launch_ctrsm_tc(float *A, int n, int lda, int64_t strideA, int batch, int *info, int c0,
                    cudaStream_t stream, bool upper)
{
    return upper ? launch_t<true>(A, n, lda, strideA, batch, info, c0, stream)
                 : launch_t<false>(A, n, lda, strideA, batch, info, c0, stream);
}

}  // namespace bl
