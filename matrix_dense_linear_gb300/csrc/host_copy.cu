// Lower-triangle copies between two buffers of the same strided-batch layout,
// for the host-buffer call on page-locked host memory the device maps: the
// batch's lower triangles go host -> device before the factorization and the
// factors device -> host after it, each element once each way, so the host
// link carries half the bytes of copying every matrix's whole span (the upper
// triangles and the gaps are not read or written on either side). One warp per
// column segment (rows j..n-1 of column j), 16-byte accesses in its aligned
// middle when both buffers start on a 16-byte boundary; the copy back also
// carries the slice's info entries.
#include "bl_common.cuh"
#include "launch.cuh"

namespace bl {
namespace {

template <bool VEC>
__global__ void __launch_bounds__(256)
tri_copy_kernel(const float *__restrict__ src, float *__restrict__ dst, int n, int lda,
                int64_t strideA, int nb, const int *__restrict__ info_src,
                int *__restrict__ info_dst)
{
    const int warps = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t cols = (int64_t)nb * n;
    for (int64_t c = (int64_t)blockIdx.x * warps + w; c < cols; c += (int64_t)gridDim.x * warps) {
        const int64_t b = c / n;
        const int j = (int)(c - b * n);
        const int64_t e0 = b * strideA + (int64_t)j * lda + j;  // first element: (j, j)
        const int64_t e1 = e0 + (n - j);                        // one past (n - 1, j)
        if constexpr (VEC) {
            int64_t a0 = (e0 + 3) & ~(int64_t)3;
            if (a0 > e1) a0 = e1;
            int64_t a1 = e1 & ~(int64_t)3;
            if (a1 < a0) a1 = a0;
            if (e0 + lane < a0) dst[e0 + lane] = src[e0 + lane];
            // four 16-byte loads a lane in flight before their stores
            for (int64_t q = a0 + 4 * lane; q < a1; q += 4 * 128) {
                float4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (q + 128 * u < a1) v[u] = *reinterpret_cast<const float4 *>(src + q + 128 * u);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (q + 128 * u < a1) *reinterpret_cast<float4 *>(dst + q + 128 * u) = v[u];
            }
            if (a1 + lane < e1) dst[a1 + lane] = src[a1 + lane];
        } else {
            for (int64_t q = e0 + lane; q < e1; q += 32) dst[q] = src[q];
        }
    }
    if (info_src != nullptr && blockIdx.x == 0)
        for (int b = threadIdx.x; b < nb; b += blockDim.x) info_dst[b] = info_src[b];
}

}  // namespace

int launch_tri_copy(const float *src, float *dst, int n, int lda, int64_t strideA, int nb,
                    const int *info_src, int *info_dst, cudaStream_t stream)
{
    if (nb <= 0) return 0;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
    // four blocks an SM at most: requests enough in flight for the host link
    // (its latency is microseconds), the rest of the SM for the factorizations
    // of the other slices
    const int64_t cols = (int64_t)nb * n;
    const int64_t need = (cols + 7) / 8;
    const int64_t cap = 4 * (int64_t)sms;
    const unsigned grid = (unsigned)(need < cap ? (need > 0 ? need : 1) : cap);
    const bool vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0;
    if (vec)
        tri_copy_kernel<true><<<grid, 256, 0, stream>>>(src, dst, n, lda, strideA, nb, info_src,
                                                       info_dst);
    else
        tri_copy_kernel<false><<<grid, 256, 0, stream>>>(src, dst, n, lda, strideA, nb, info_src,
                                                        info_dst);
    return (int)cudaGetLastError();
}

}  // namespace bl
