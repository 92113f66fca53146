// Pieces of the shared-memory kernel for n <= 128 (K2): the packed panel
// storage of the lower triangle, its bulk copies, the warp-level diagonal
// factor and the one-row panel solve.
#pragma once

#include "bl_common.cuh"
#include "tc_sm100.cuh"

namespace bl {
namespace cta {

constexpr int kPad = 4;
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s

template <int NB>
struct CtaGeom {
    static constexpr int NP = 32 * NB;
    __host__ __device__ static constexpr int ld(int p) { return NP - 32 * p + kPad; }
    __host__ __device__ static constexpr int off(int p) {
        // sum_{q<p} 32 * ld(q)
        return 32 * (p * (NP + kPad) - 32 * (p * (p - 1) / 2));
    }
    static constexpr int floats = off(NB);
    static constexpr int bytes = floats * 4;
};

template <int NB>
__device__ __forceinline__ float *elem_ptr(float *S, int i, int k)
{
    // address of element (i, k), i >= 32*(k/32), in the packed storage
    using Gm = CtaGeom<NB>;
    const int p = k >> 5;
    return S + Gm::off(p) + (i - 32 * p) + (k - 32 * p) * Gm::ld(p);
}

// Step 1: factor the diagonal block of panel p in one warp, lane = row, with
// the broadcast-column step of K1. P points at element (c0, c0); ldp is the
// panel's leading dimension. Per column j every lane publishes r[j] to a
// warp-private buffer, one __syncwarp, and reads the pivot d_j and the column
// below it back as 16-byte broadcasts (from the quad holding d_j on); then
// l = r[j] rsqrt(d_j) and r[k] -= (l rsqrt(d_j)) c_k for k > j. Lane j keeps
// its pivot; at the end every lane writes s = rsqrt(d) of its column to sinv
// and the first pivot with !(d > 0) is reported as c0 + j + 1 in *fail_out;
// the diagonal entry is sqrt(d_j). Columns from n on (the identity block) are
// left as they are.
__device__ __forceinline__ void factor_diag_block(float *P, int ldp, int lane, int c0, int n,
                                                  float (*colbuf)[32], float *sinv,
                                                  int *fail_out)
{
    float r[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) r[k] = P[lane + k * ldp];
    float my_d = 1.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        if (c0 + j >= n) break;
        float *cb = colbuf[j & 1];
        cb[lane] = r[j];
        __syncwarp();
        const float4 f4 = reinterpret_cast<const float4 *>(cb)[j / 4];
        const float fv[4] = {f4.x, f4.y, f4.z, f4.w};
        const float d = fv[j % 4];
        my_d = (lane == j) ? d : my_d;
        const float s = rsqrt_approx(d);
        const float lij = r[j] * s;
        const float w = lij * s;
        r[j] = lij;
#pragma unroll
        for (int t = j % 4 + 1; t < 4; ++t) r[4 * (j / 4) + t] = fmaf(-w, fv[t], r[4 * (j / 4) + t]);
        const float2 nw = make_float2(-w, -w);
#pragma unroll
        for (int q = j / 4 + 1; q < 8; ++q) {
            const float4 c4 = reinterpret_cast<const float4 *>(cb)[q];
            float2 t0 = __ffma2_rn(nw, make_float2(c4.x, c4.y), make_float2(r[4 * q], r[4 * q + 1]));
            float2 t1 = __ffma2_rn(nw, make_float2(c4.z, c4.w), make_float2(r[4 * q + 2], r[4 * q + 3]));
            r[4 * q] = t0.x; r[4 * q + 1] = t0.y; r[4 * q + 2] = t1.x; r[4 * q + 3] = t1.y;
        }
    }
#pragma unroll
    for (int k = 0; k < 32; ++k)
        if (k < lane) P[lane + k * ldp] = r[k];
    // the diagonal from the lane's own pivot (sqrt(+Inf) = +Inf, like the definition)
    if (c0 + lane < n) P[lane + lane * ldp] = sqrt_approx(my_d);
    sinv[lane] = rsqrt_approx(my_d);
    const unsigned bad = __ballot_sync(0xffffffffu, !pivot_ok(my_d));
    if (lane == 0 && bad) *fail_out = c0 + __ffs(bad);
}

// Step 2: row a (>= 32, panel coordinates) of panel p: x <- x L11^{-T}, with
// L11 the panel's factored diagonal block and sinv its reciprocal diagonal;
// the solved row is stored back and left in x. Here and in step 1 the updates
// go by pairs of columns through the paired single-precision FMA.
__device__ __forceinline__ void trsm_row_x(float *P, int ldp, int a, const float *sinv,
                                           float (&x)[32])
{
#pragma unroll
    for (int k = 0; k < 32; ++k) x[k] = P[a + k * ldp];
    float4 s4;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        if (j % 4 == 0) s4 = reinterpret_cast<const float4 *>(sinv)[j / 4];
        x[j] *= (j % 4 == 0) ? s4.x : (j % 4 == 1) ? s4.y : (j % 4 == 2) ? s4.z : s4.w;
        const float *Lj = P + j * ldp;  // column j of L11, rows 0..31
        const float2 nx = make_float2(-x[j], -x[j]);
#pragma unroll
        for (int q = (j + 1) / 4; q < 8; ++q) {
            const float4 l4 = reinterpret_cast<const float4 *>(Lj)[q];
            const float2 lp[2] = {make_float2(l4.x, l4.y), make_float2(l4.z, l4.w)};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int k = 4 * q + 2 * h;
                if (k > j) {
                    const float2 t = __ffma2_rn(nx, lp[h], make_float2(x[k], x[k + 1]));
                    x[k] = t.x; x[k + 1] = t.y;
                } else if (k + 1 > j) {
                    x[k + 1] = fmaf(-x[j], lp[h].y, x[k + 1]);
                }
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 32; ++k) P[a + k * ldp] = x[k];
}

__device__ __forceinline__ void trsm_row(float *P, int ldp, int a, const float *sinv)
{
    float x[32];
    trsm_row_x(P, ldp, a, sinv, x);
}

// The same two copies for the common exact case n = NP with 16-byte aligned
// columns, by the bulk-copy engine: thread k moves column k, rows ceil4(k) ..
// NP-1 as one bulk copy (16-byte aligned on both sides) and its 0-3 leading
// rows k .. ceil4(k)-1 with plain loads and stores. Loads complete on mbar[0]
// (columns 0..31, arrival count 32) and mbar[1] (the rest, NP-32).
template <int NB>
__device__ __forceinline__ void bulk_load_full(float *S, const float *Ab, int lda, int tid,
                                               uint64_t *mbar)
{
    constexpr int NP = CtaGeom<NB>::NP;
    if (tid >= NP) return;
    const int k = tid, q0 = (k + 3) & ~3;
    const float *g = Ab + (int64_t)k * lda;
    float *col = elem_ptr<NB>(S, 0, k);  // col[i] = element (i, k)
    uint64_t *bar = mbar + (k < 32 ? 0 : 1);
    const uint32_t bytes = 4u * (uint32_t)(NP - q0);
    tc::mbar_arrive_expect_tx(bar, bytes);
    if (bytes) tc::bulk_g2s(col + q0, g + q0, bytes, bar);
    const int m = q0 - k;  // 0..3 leading rows (q0 <= NP)
    if (m > 0) col[k] = g[k];
    if (m > 1) col[k + 1] = g[k + 1];
    if (m > 2) col[k + 2] = g[k + 2];
}

template <int NB>
__device__ __forceinline__ void bulk_store_full(const float *S, float *Ab, int lda, int tid)
{
    constexpr int NP = CtaGeom<NB>::NP;
    if (tid >= NP) return;
    const int k = tid, q0 = (k + 3) & ~3;
    float *g = Ab + (int64_t)k * lda;
    const float *col = elem_ptr<NB>(const_cast<float *>(S), 0, k);
    const uint32_t bytes = 4u * (uint32_t)(NP - q0);
    if (bytes) {
        tc::bulk_s2g(g + q0, col + q0, bytes);
        tc::bulk_commit();
    }
    const int m = q0 - k;
    if (m > 0) g[k] = col[k];
    if (m > 1) g[k + 1] = col[k + 1];
    if (m > 2) g[k + 2] = col[k + 2];
    if (bytes) tc::bulk_wait_read0();  // the block's shared memory outlives the reads
}

}  // namespace cta
}  // namespace bl
