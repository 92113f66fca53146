// FMA-throughput probe: the FP32 and FP64 rates this device reaches with
// independent FMA chains on every SM, the denominators the measurement of the
// factorizations is read against (the FP32 roofline is the unit count times
// the clock; the FP64 rate of this GPU is measured here).
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bl_spotrf.h"

namespace {

template <typename T>
__global__ void __launch_bounds__(256) fma_probe_kernel(T *out, int iters)
{
    // eight independent chains a thread
    T a[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) a[c] = (T)(threadIdx.x + c) * (T)1e-3;
    const T b = (T)0.999, d = (T)1e-7;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < 8; ++c) a[c] = a[c] * b + d;
    }
    T s = 0;
#pragma unroll
    for (int c = 0; c < 8; ++c) s += a[c];
    if (s == (T)-1) out[0] = s;  // never true; keeps the chains alive
}

template <typename T>
int run(T *out, double *tflops, cudaStream_t st)
{
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)))
        return (int)e;
    const int blocks = 8 * sms, threads = 256;
    const int iters = sizeof(T) == 8 ? 2000 : 20000;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if ((e = cudaEventCreate(&e0)) || (e = cudaEventCreate(&e1))) return (int)e;
    fma_probe_kernel<T><<<blocks, threads, 0, st>>>(out, 10);  // warm-up
    cudaEventRecord(e0, st);
    fma_probe_kernel<T><<<blocks, threads, 0, st>>>(out, iters);
    cudaEventRecord(e1, st);
    e = cudaGetLastError();
    if (!e) e = cudaEventSynchronize(e1);
    float ms = 0.0f;
    if (!e) e = cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (e) return (int)e;
    const double flops = 2.0 * 8 * (double)iters * blocks * threads;
    *tflops = ms > 0.0f ? flops / (ms * 1e-3) / 1e12 : 0.0;
    return 0;
}

}  // namespace

extern "C" int bl_fma_probe(int precision, void *out, double *tflops, cudaStream_t stream)
{
    if (precision != 32 && precision != 64) return -1;
    if (out == nullptr) return -2;
    if (tflops == nullptr) return -3;
    return precision == 64 ? run(static_cast<double *>(out), tflops, stream)
                           : run(static_cast<float *>(out), tflops, stream);
}
