// Throughput probe of the FP32 FFMA pipes: the denominator of the SGEMM's
// roofline measured instead of derived.  The m.lqnn.cn SGEMM article
// (sections 1.1-1.2) states a kernel's efficiency against the card's FP32
// peak and its arithmetic intensity; the peak here is what the SMs' FMA
// pipes deliver at the clock the probe runs at, timed by the caller.
//
// Every thread keeps kChains independent packed accumulators and applies
// one fma.rn.f32x2 (two FP32 FMAs, four FLOPs) to each per iteration, so
// the FMA pipe never waits for a result; nothing is loaded or stored
// except one value per thread at the end (so the work is not removed).
#include <cstdint>

#include <cuda_runtime.h>

#include "dense_gemm.h"
#include "launch.h"

namespace {

constexpr int kChains = 16;          // independent FFMA2 chains per thread
constexpr int kProbeThreads = 256;

__device__ __forceinline__ void ffma2(unsigned long long& d, unsigned long long a,
                                      unsigned long long b) {
  asm volatile("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

__global__ void __launch_bounds__(kProbeThreads)
    ffma2_probe_kernel(int iters, float x, float y, float* __restrict__ out) {
  unsigned long long acc[kChains];
  const float seed = (float)(threadIdx.x + blockIdx.x) * 1e-7f;
#pragma unroll
  for (int i = 0; i < kChains; ++i) {
    const float v = seed + (float)i * 1e-6f;
    acc[i] = ((unsigned long long)__float_as_uint(v) << 32) | __float_as_uint(v);
  }
  const unsigned long long a = ((unsigned long long)__float_as_uint(x) << 32) | __float_as_uint(x);
  const unsigned long long b = ((unsigned long long)__float_as_uint(y) << 32) | __float_as_uint(y);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < kChains; ++i) ffma2(acc[i], a, b);
  }
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < kChains; ++i)
    sum += __uint_as_float((unsigned)acc[i]) + __uint_as_float((unsigned)(acc[i] >> 32));
  out[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = sum;
}

}  // namespace

extern "C" gemm_status_t gemm_probe_ffma(int blocks, int iters, float* out, cudaStream_t stream,
                                         double* flops) {
  if (blocks <= 0 || iters <= 0 || out == nullptr) return GEMM_ERR_INVALID_ARG;
  if (flops != nullptr)
    *flops = (double)blocks * kProbeThreads * (double)iters * kChains * 4.0;
  // x * y + acc with |x * y| < 1 keeps every value finite and normal.
  ffma2_probe_kernel<<<blocks, kProbeThreads, 0, stream>>>(iters, 0.999f, 1e-3f, out);
  if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;
  return GEMM_OK;
}

extern "C" int gemm_probe_ffma_threads(void) { return kProbeThreads; }
