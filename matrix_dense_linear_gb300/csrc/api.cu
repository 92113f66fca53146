// C-ABI of libbl_spotrf: argument checks, the size-keyed route selector and
// the quick returns. Declarations and the contract are in include/bl_spotrf.h.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "../../include/bl_spotrf.h"
#include "bl_common.cuh"
#include "launch.cuh"

namespace {

// Size thresholds of the selector. The pages route by order the same way
// (one warp per matrix up to n = 32, one work-group per matrix in the middle,
// blocked above: "BatchLAS perf_blackwell", potrf row of its routing table;
// the size router of "kernelbot-cholesky-930185"). Measured on GB300: the
// register-resident warp kernel wins up to n = 64; for 65..128 the shared-
// memory block kernel (K2) beats the tensor-memory one (K2t, reachable as a
// forced route) at 1024 matrices of n = 128 (about 70 us against 89 us).
constexpr int kWarpMaxN = 64;
constexpr int kCtaMaxN = 128;

bool trace_enabled()
{
    static std::once_flag once;
    static bool on = false;
    std::call_once(once, [] {
        const char *v = std::getenv("BL_TRACE");
        on = v && *v && *v != '0';
    });
    return on;
}

int check_args(const void *A, int n, int lda, int64_t strideA, int batch, const int *info)
{
    if (n < 0) return -2;
    if (batch < 0) return -5;
    if (lda < (n > 1 ? n : 1)) return -3;
    if (batch > 1 && strideA < (int64_t)lda * n) return -4;
    if (A == nullptr && n > 0 && batch > 0) return -1;
    if (info == nullptr && batch > 0) return -6;
    if (n > BL_SPOTRF_MAX_N) return -7;
    return 0;
}

int route_for(int n)
{
    if (n <= kWarpMaxN) return BL_ROUTE_WARP;
    if (n <= kCtaMaxN) return BL_ROUTE_CTA;
    return BL_ROUTE_BLOCKED;
}

bool route_can_run(int route, int n, bool upper)
{
    switch (route) {
    case BL_ROUTE_WARP: return n <= kWarpMaxN;
    case BL_ROUTE_CTA: return n <= kCtaMaxN;
    case BL_ROUTE_TMEM: return n <= kCtaMaxN && !upper;
    case BL_ROUTE_BLOCKED: return true;
    case BL_ROUTE_LEFT: return n > kCtaMaxN;
    default: return false;
    }
}

int run(float *A, int n, int lda, int64_t strideA, int batch, int *info, cudaStream_t stream,
        int route, bool upper = false, bool host_mapped = false, float *W = nullptr)
{
    int e = check_args(A, n, lda, strideA, batch, info);
    if (e) return e;
    if (route == BL_ROUTE_AUTO) {
        route = route_for(n);
        // large batches of 16-byte-aligned matrices without a workspace: the
        // blocked route's kernels in the left-looking order (a forced
        // BL_ROUTE_BLOCKED keeps the right-looking one)
        const bool aligned = ((reinterpret_cast<uintptr_t>(A) & 15) == 0) && (lda & 3) == 0 &&
                             (strideA & 3) == 0;
        if (route == BL_ROUTE_BLOCKED && W == nullptr && aligned &&
            bl::left_pays(n, batch, bl::sm_count_or_default()))
            route = BL_ROUTE_LEFT;
    }
    if (!route_can_run(route, n, upper)) return -8;
    if (batch == 0) return 0;
    if (n == 0) return (int)cudaMemsetAsync(info, 0, sizeof(int) * (size_t)batch, stream);
    if (trace_enabled())
        std::fprintf(stderr, "bl_spotrf: uplo=%c n=%d lda=%d strideA=%lld batch=%d route=%d\n",
                     upper ? 'U' : 'L', n, lda, (long long)strideA, batch, route);
    switch (route) {
    case BL_ROUTE_WARP: return bl::launch_warp(A, n, lda, strideA, batch, info, stream, upper);
    case BL_ROUTE_CTA:
        return bl::launch_cta(A, n, lda, strideA, batch, info, stream, bl::InfoMode{-1}, upper,
                              host_mapped);
    case BL_ROUTE_TMEM:
        return bl::launch_tmem(A, n, lda, strideA, batch, info, stream, bl::InfoMode{-1});
    case BL_ROUTE_LEFT: return bl::launch_left(A, n, lda, strideA, batch, info, stream, upper);
    default: return bl::launch_blocked(A, n, lda, strideA, batch, info, stream, upper, W);
    }
}

// Workspace of the inverse-based panel solve: one 128 x 128 block per matrix
// on the blocked route (n > 128), none below.
size_t workspace_bytes(int n, int batch)
{
    if (n <= kCtaMaxN || n > BL_SPOTRF_MAX_N || batch <= 0) return 0;
    return bl::kInvBytes * (size_t)batch;
}

// the calls with a workspace: the argument checks of run(), then work (-8: not
// 16-byte aligned; -9: work_bytes too small), then run()
int run_ws(float *A, int n, int lda, int64_t strideA, int batch, int *info, void *work,
           size_t work_bytes, cudaStream_t stream, bool upper)
{
    int e = check_args(A, n, lda, strideA, batch, info);
    if (e) return e;
    if (work != nullptr) {
        if ((reinterpret_cast<uintptr_t>(work) & 15) != 0) return -8;
        if (work_bytes < workspace_bytes(n, batch)) return -9;
    }
    return run(A, n, lda, strideA, batch, info, stream, BL_ROUTE_AUTO, upper, false,
               static_cast<float *>(work));
}

// The device address of a page-locked host allocation the device maps (with
// unified addressing every cudaHostAlloc / cudaHostRegister allocation is),
// else nullptr (pageable memory, device memory, or no information).
template <typename T>
T *mapped_host(T *p)
{
    cudaPointerAttributes at{};
    if (p == nullptr || cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // clear a failed query
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return nullptr;
    return static_cast<T *>(at.devicePointer);
}

// uplo argument: 0 lower, 1 upper, -1 invalid
int parse_uplo(char uplo)
{
    if (uplo == 'L' || uplo == 'l') return 0;
    if (uplo == 'U' || uplo == 'u') return 1;
    return -1;
}

// the uplo entry points take uplo as argument 1: every other argument index
// moves up by one
int shift_arg(int e) { return e < 0 ? e - 1 : e; }

int check_trs_args(const float *L, int n, int lda, int64_t strideA, const float *B, int nrhs,
                   int ldb, int64_t strideB, int batch)
{
    if (n < 0 || n > BL_SPOTRF_MAX_N) return -2;
    if (nrhs < 0) return -6;
    if (batch < 0) return -9;
    if (lda < (n > 1 ? n : 1)) return -3;
    if (ldb < (n > 1 ? n : 1)) return -7;
    if (batch > 1 && strideA < (int64_t)lda * n) return -4;
    if (batch > 1 && strideB < (int64_t)ldb * nrhs) return -8;
    const bool work = n > 0 && nrhs > 0 && batch > 0;
    if (work && L == nullptr) return -1;
    if (work && B == nullptr) return -5;
    return 0;
}

}  // namespace

// the argument checks of bl_spotrf_batched, for entry points in other files
int bl::check_potrf_args(const void *A, int n, int lda, int64_t strideA, int batch,
                         const int *info)
{
    return check_args(A, n, lda, strideA, batch, info);
}

extern "C" {

int bl_spotrf_batched_host(float *A_host, int n, int lda, int64_t strideA, int batch,
                           int *info_host, float *A_dev, int *info_dev, int chunks,
                           const cudaStream_t *streams, int nstreams)
{
    int e = check_args(A_dev, n, lda, strideA, batch, info_dev);
    if (e) return e;
    if (batch > 0 && n > 0 && A_host == nullptr) return -1;
    if (batch > 0 && info_host == nullptr) return -6;
    if (streams == nullptr || nstreams < 1) return -11;
    if (batch == 0) return 0;
    // Page-locked host buffers of a one-kernel order (n <= 128): the kernel
    // reads and writes them in place over the host link (lower triangles only,
    // each element once each way), with no staging copies; on GB300 the
    // NVLink-C2C link carries that at about 1.5 times the rate of the copy
    // engines (1024 matrices of order 64: 137 against 207 us).
    float *Am = n > 0 ? mapped_host(A_host) : nullptr;
    int *im = mapped_host(info_host);
    if (n <= kCtaMaxN && Am && im)
        return run(Am, n, lda, strideA, batch, im, streams[0], BL_ROUTE_AUTO, false, true);
    // Larger orders on such buffers: per slice, a kernel copies the lower
    // triangles host -> device, the slice is factored, a kernel copies the
    // factors and info back: half the bytes of whole spans, each way. Issued
    // slice by slice (four a stream unless chunks says otherwise), so that one
    // stream's copy in runs while another's copy back does and the link
    // carries both directions at once.
    if (Am && im) {
        if (chunks <= 0) chunks = 4 * nstreams;
        if (chunks > batch) chunks = batch;
        for (int c = 0; c < chunks; ++c) {
            const int b0 = (int)((int64_t)batch * c / chunks);
            const int b1 = (int)((int64_t)batch * (c + 1) / chunks);
            if (b1 <= b0) continue;
            cudaStream_t s = streams[c % nstreams];
            const int64_t off = (int64_t)b0 * strideA;
            if ((e = bl::launch_tri_copy(Am + off, A_dev + off, n, lda, strideA, b1 - b0, nullptr,
                                         nullptr, s)))
                return e;
            if ((e = run(A_dev + off, n, lda, strideA, b1 - b0, info_dev + b0, s, BL_ROUTE_AUTO)))
                return e;
            if ((e = bl::launch_tri_copy(A_dev + off, Am + off, n, lda, strideA, b1 - b0,
                                         info_dev + b0, im + b0, s)))
                return e;
        }
        return 0;
    }
    const int64_t span = (int64_t)lda * n;  // floats of one matrix
    if (chunks <= 0) chunks = nstreams;
    if (chunks > batch) chunks = batch;
    // Issued phase by phase (every slice's copy in, then every factorization,
    // then every copy out): a copy out waits for its factorization, and copies
    // queued behind it would wait too, so the copies in go first.
    for (int phase = 0; phase < 3; ++phase) {
        for (int c = 0; c < chunks; ++c) {
            const int b0 = (int)((int64_t)batch * c / chunks);
            const int b1 = (int)((int64_t)batch * (c + 1) / chunks);
            if (b1 <= b0) continue;
            cudaStream_t s = streams[c % nstreams];
            const int64_t off = (int64_t)b0 * strideA;
            const size_t bytes = (size_t)(((int64_t)(b1 - 1 - b0) * strideA + span) * 4);
            if (phase == 0 && n > 0)
                e = (int)cudaMemcpyAsync(A_dev + off, A_host + off, bytes, cudaMemcpyHostToDevice,
                                         s);
            else if (phase == 1)
                e = run(A_dev + off, n, lda, strideA, b1 - b0, info_dev + b0, s, BL_ROUTE_AUTO);
            else if (phase == 2) {
                if (n > 0)
                    e = (int)cudaMemcpyAsync(A_host + off, A_dev + off, bytes,
                                             cudaMemcpyDeviceToHost, s);
                if (!e)
                    e = (int)cudaMemcpyAsync(info_host + b0, info_dev + b0,
                                             sizeof(int) * (size_t)(b1 - b0),
                                             cudaMemcpyDeviceToHost, s);
            }
            if (e) return e;
        }
    }
    return 0;
}

}  // extern "C"

namespace {

int spotrs(bool upper, const float *L, int n, int lda, int64_t strideA, float *B, int nrhs,
           int ldb, int64_t strideB, int batch, cudaStream_t stream)
{
    const int e = check_trs_args(L, n, lda, strideA, B, nrhs, ldb, strideB, batch);
    if (e) return e;
    if (batch == 0 || n == 0 || nrhs == 0) return 0;
    if (trace_enabled())
        std::fprintf(stderr, "bl_spotrs: uplo=%c n=%d nrhs=%d batch=%d\n", upper ? 'U' : 'L', n,
                     nrhs, batch);
    return bl::launch_potrs(L, n, lda, strideA, B, nrhs, ldb, strideB, batch, nullptr, stream,
                            upper);
}

int sposv(bool upper, float *A, int n, int lda, int64_t strideA, float *B, int nrhs, int ldb,
          int64_t strideB, int batch, int *info, cudaStream_t stream)
{
    int e = check_trs_args(A, n, lda, strideA, B, nrhs, ldb, strideB, batch);
    if (e) return e;
    if (info == nullptr && batch > 0) return -10;
    e = run(A, n, lda, strideA, batch, info, stream, BL_ROUTE_AUTO, upper);
    if (e || batch == 0 || n == 0 || nrhs == 0) return e;
    return bl::launch_potrs(A, n, lda, strideA, B, nrhs, ldb, strideB, batch, info, stream,
                            upper);
}

}  // namespace

extern "C" {

int bl_spotrs_batched(const float *L, int n, int lda, int64_t strideA, float *B, int nrhs,
                      int ldb, int64_t strideB, int batch, cudaStream_t stream)
{
    return spotrs(false, L, n, lda, strideA, B, nrhs, ldb, strideB, batch, stream);
}

int bl_sposv_batched(float *A, int n, int lda, int64_t strideA, float *B, int nrhs, int ldb,
                     int64_t strideB, int batch, int *info, cudaStream_t stream)
{
    return sposv(false, A, n, lda, strideA, B, nrhs, ldb, strideB, batch, info, stream);
}

int bl_spotrs_batched_uplo(char uplo, const float *A, int n, int lda, int64_t strideA, float *B,
                           int nrhs, int ldb, int64_t strideB, int batch, cudaStream_t stream)
{
    const int u = parse_uplo(uplo);
    if (u < 0) return -1;
    return shift_arg(spotrs(u == 1, A, n, lda, strideA, B, nrhs, ldb, strideB, batch, stream));
}

int bl_sposv_batched_uplo(char uplo, float *A, int n, int lda, int64_t strideA, float *B,
                          int nrhs, int ldb, int64_t strideB, int batch, int *info,
                          cudaStream_t stream)
{
    const int u = parse_uplo(uplo);
    if (u < 0) return -1;
    return shift_arg(sposv(u == 1, A, n, lda, strideA, B, nrhs, ldb, strideB, batch, info,
                           stream));
}

int bl_spotrf_batched_uplo(char uplo, float *A, int n, int lda, int64_t strideA, int batch,
                           int *info, cudaStream_t stream)
{
    const int u = parse_uplo(uplo);
    if (u < 0) return -1;
    return shift_arg(run(A, n, lda, strideA, batch, info, stream, BL_ROUTE_AUTO, u == 1));
}

int bl_dpotrf_batched_uplo(char uplo, double *A, int n, int lda, int64_t strideA, int batch,
                           int *info, cudaStream_t stream)
{
    const int u = parse_uplo(uplo);
    if (u < 0) return -1;
    const int e = check_args(A, n, lda, strideA, batch, info);
    if (e) return shift_arg(e);
    if (batch == 0) return 0;
    if (n == 0) return (int)cudaMemsetAsync(info, 0, sizeof(int) * (size_t)batch, stream);
    if (trace_enabled())
        std::fprintf(stderr, "bl_dpotrf: uplo=%c n=%d lda=%d strideA=%lld batch=%d\n",
                     u ? 'U' : 'L', n, lda, (long long)strideA, batch);
    return bl::launch_dpotrf(A, n, lda, strideA, batch, info, stream, u == 1);
}

int bl_cpotrf_batched_uplo(char uplo, float *A, int n, int lda, int64_t strideA, int batch,
                           int *info, cudaStream_t stream)
{
    const int u = parse_uplo(uplo);
    if (u < 0) return -1;
    const int e = check_args(A, n, lda, strideA, batch, info);
    if (e) return shift_arg(e);
    if (batch > 0 && n > 0 && (reinterpret_cast<uintptr_t>(A) & 7) != 0) return -2;
    if (batch == 0) return 0;
    if (n == 0) return (int)cudaMemsetAsync(info, 0, sizeof(int) * (size_t)batch, stream);
    if (trace_enabled())
        std::fprintf(stderr, "bl_cpotrf: uplo=%c n=%d lda=%d strideA=%lld batch=%d\n",
                     u ? 'U' : 'L', n, lda, (long long)strideA, batch);
    return bl::launch_cpotrf(A, n, lda, strideA, batch, info, stream, u == 1);
}

int bl_cpotrf_batched(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                      cudaStream_t stream)
{
    const int e = bl_cpotrf_batched_uplo('L', A, n, lda, strideA, batch, info, stream);
    return e < 0 ? e + 1 : e;
}

int bl_zpotrf_batched_uplo(char uplo, double *A, int n, int lda, int64_t strideA, int batch,
                           int *info, cudaStream_t stream)
{
    const int u = parse_uplo(uplo);
    if (u < 0) return -1;
    const int e = check_args(A, n, lda, strideA, batch, info);
    if (e) return shift_arg(e);
    if (batch > 0 && n > 0 && (reinterpret_cast<uintptr_t>(A) & 15) != 0) return -2;
    if (batch == 0) return 0;
    if (n == 0) return (int)cudaMemsetAsync(info, 0, sizeof(int) * (size_t)batch, stream);
    if (trace_enabled())
        std::fprintf(stderr, "bl_zpotrf: uplo=%c n=%d lda=%d strideA=%lld batch=%d\n",
                     u ? 'U' : 'L', n, lda, (long long)strideA, batch);
    return bl::launch_zpotrf(A, n, lda, strideA, batch, info, stream, u == 1);
}

int bl_zpotrf_batched(double *A, int n, int lda, int64_t strideA, int batch, int *info,
                      cudaStream_t stream)
{
    const int e = bl_zpotrf_batched_uplo('L', A, n, lda, strideA, batch, info, stream);
    return e < 0 ? e + 1 : e;
}

int bl_dpotrf_batched(double *A, int n, int lda, int64_t strideA, int batch, int *info,
                      cudaStream_t stream)
{
    const int e = bl_dpotrf_batched_uplo('L', A, n, lda, strideA, batch, info, stream);
    return e < 0 ? e + 1 : e;  // argument indices without the uplo argument
}

int bl_spotrf_batched_uplo_ex(char uplo, float *A, int n, int lda, int64_t strideA, int batch,
                              int *info, cudaStream_t stream, int route)
{
    const int u = parse_uplo(uplo);
    if (u < 0) return -1;
    if (route < BL_ROUTE_AUTO || route > BL_ROUTE_LEFT) return -9;
    return shift_arg(run(A, n, lda, strideA, batch, info, stream, route, u == 1));
}


int bl_spotrf_batched(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                      cudaStream_t stream)
{
    return run(A, n, lda, strideA, batch, info, stream, BL_ROUTE_AUTO);
}

int bl_spotrf_batched_ex(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                         cudaStream_t stream, int route)
{
    if (route < BL_ROUTE_AUTO || route > BL_ROUTE_LEFT) return -8;
    return run(A, n, lda, strideA, batch, info, stream, route);
}

int bl_spotrf_route(int n, int batch)
{
    if (n <= 0 || batch <= 0) return 0;
    const int r = route_for(n);
    if (r == BL_ROUTE_BLOCKED && n <= BL_SPOTRF_MAX_N &&
        bl::left_pays(n, batch, bl::sm_count_or_default()))
        return BL_ROUTE_LEFT;
    return r;
}

int bl_spotrf_kernel_info(int route, int n, int *regs, int *local_bytes, int *static_smem,
                          int *dynamic_smem, int *threads)
{
    if (route == BL_ROUTE_AUTO) route = route_for(n);
    if (n < 1 || !route_can_run(route, n, false)) return -8;
    cudaFuncAttributes fa{};
    int th = 0, dyn = 0, e;
    switch (route) {
    case BL_ROUTE_WARP: e = bl::attrs_warp(n, &fa, &th, &dyn); break;
    case BL_ROUTE_CTA: e = bl::attrs_cta(n, &fa, &th, &dyn); break;
    case BL_ROUTE_TMEM: e = bl::attrs_tmem(n, &fa, &th, &dyn); break;
    default: e = bl::attrs_blocked(n, &fa, &th, &dyn); break;
    }
    if (e) return e;
    if (regs) *regs = fa.numRegs;
    if (local_bytes) *local_bytes = (int)fa.localSizeBytes;
    if (static_smem) *static_smem = (int)fa.sharedSizeBytes;
    if (dynamic_smem) *dynamic_smem = dyn;
    if (threads) *threads = th;
    return 0;
}

size_t bl_spotrf_workspace_bytes(int n, int batch) { return workspace_bytes(n, batch); }

int bl_spotrf_batched_ws(float *A, int n, int lda, int64_t strideA, int batch, int *info,
                         void *work, size_t work_bytes, cudaStream_t stream)
{
    return run_ws(A, n, lda, strideA, batch, info, work, work_bytes, stream, false);
}

int bl_spotrf_batched_uplo_ws(char uplo, float *A, int n, int lda, int64_t strideA, int batch,
                              int *info, void *work, size_t work_bytes, cudaStream_t stream)
{
    const int u = parse_uplo(uplo);
    if (u < 0) return -1;
    return shift_arg(run_ws(A, n, lda, strideA, batch, info, work, work_bytes, stream, u == 1));
}

int bl_debug_fail_first_wait(int kernel_class, int every)
{
    if (every < 0) return -2;
    switch (kernel_class) {
    case 1: return bl::set_fail_first_wait_cta(every);
    case 2: return bl::set_fail_first_wait_trsm_tc(every);
    case 3: return bl::set_fail_first_wait_syrk_tc(every);
    case 4: return bl::set_fail_first_wait_tmem(every);
    case 5: return bl::set_fail_first_wait_trsm_inv(every);
    case 6: return bl::set_fail_first_wait_cherk_tc(every);
    case 7: return bl::set_fail_first_wait_ctrsm_tc(every);
    default: return -1;
    }
}

const char *bl_spotrf_version(void) { return "bl_spotrf 0.2 sm_103a"; }

}  // extern "C"
