// bl_spotrf_batched_static: the factorization of bl_spotrf_batched_ws with its
// workspace taken from a fixed array of device memory that the library
// reserves when it is loaded, so that the call itself allocates nothing.
//
// Who needs it: callers that cannot allocate device memory where they factor.
// A library called from inside a framework that manages all device memory
// through its own allocator cannot reach that allocator; a latency-bounded
// loop cannot afford the device-wide synchronization that cudaMalloc and
// cudaFree may bring; a process may already hold all the memory it was given.
// Those callers still pass A and info; only the inverse-based panel solve's
// scratch (one 128 x 128 float block per matrix of order > 128) comes from
// here.
//
// The array is BL_SPOTRF_STATIC_SCRATCH_BYTES (16 MB) on every GPU that loads
// the library, held until the process exits; calls whose scratch would not fit
// (n > 128 and batch > 256) are rejected with -10 before any work.
#include <cstdint>
#include <mutex>

#include "../../include/bl_spotrf.h"
#include "launch.cuh"

namespace {

constexpr size_t kScratchBytes = BL_SPOTRF_STATIC_SCRATCH_BYTES;
static_assert(kScratchBytes % bl::kInvBytes == 0, "the scratch holds whole matrices' blocks");
static_assert(kScratchBytes % 256 == 0, "the scratch is a whole number of 256-byte units");

static __device__ __align__(256) float g_scratch[kScratchBytes / sizeof(float)];

// In host code g_scratch names a host-side stand-in, not device memory: the
// kernels are given the array's device address, looked up once per device,
// with that device current, by the first call made on it.
constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
float *g_addr[kMaxDevices];
cudaError_t g_err[kMaxDevices];

int scratch_address(float **out)
{
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
    std::call_once(g_once[dev], [dev] {
        void *p = nullptr;
        g_err[dev] = cudaGetSymbolAddress(&p, g_scratch);
        g_addr[dev] = g_err[dev] == cudaSuccess ? static_cast<float *>(p) : nullptr;
    });
    if (g_err[dev] != cudaSuccess) return (int)g_err[dev];
    *out = g_addr[dev];
    return 0;
}

}  // namespace

extern "C" int bl_spotrf_batched_static(float *A, int n, int lda, int64_t strideA, int batch,
                                        int *info, cudaStream_t stream)
{
    if (const int e = bl::check_potrf_args(A, n, lda, strideA, batch, info)) return e;
    const size_t need = bl_spotrf_workspace_bytes(n, batch);
    if (need > kScratchBytes) return -10;
    float *W = nullptr;
    if (need > 0) {
        if (const int e = scratch_address(&W)) return e;
    }
    // every block of the scratch that a call reads it writes first (the
    // inverse of that matrix's diagonal block), so nothing needs clearing
    return bl_spotrf_batched_ws(A, n, lda, strideA, batch, info, W, need, stream);
}
