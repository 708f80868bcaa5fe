// Small kernels around the GEMM path: the K == 0 product (C := 0) and the
// self-test of the bounded mbarrier wait.
#include "launch.h"
#include "ptx.cuh"

namespace dgemm {
namespace {

// Grid-stride zero fill of an M x N row-major block with leading dimension
// ldc; elements of a row are contiguous, rows may be padded.
template <typename T>
__global__ void zero_fill_kernel(T* C, int M, int N, long long ldc) {
  const long long total = (long long)M * N;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long i = idx / N;
    const long long j = idx - i * N;
    C[i * ldc + j] = T(0);
  }
}

// One thread waits on a freshly initialised mbarrier that expects one
// arrival which never comes.  The bounded wait gives up after timeout_ns
// and the kernel records kFaultSelftestWait.
__global__ void selftest_timeout_kernel(unsigned* fault, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  if (!mbar_wait_bounded(b, 0, timeout_ns, nullptr)) raise_fault(fault, kFaultSelftestWait);
}

}  // namespace

cudaError_t launch_zero_fill(void* C, int M, int N, long long ldc, int elem_bytes,
                             cudaStream_t stream) {
  const long long total = (long long)M * N;
  long long blocks = (total + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  if (elem_bytes == 4)
    zero_fill_kernel<float><<<(unsigned)blocks, 256, 0, stream>>>(static_cast<float*>(C), M, N, ldc);
  else
    zero_fill_kernel<unsigned short>
        <<<(unsigned)blocks, 256, 0, stream>>>(static_cast<unsigned short*>(C), M, N, ldc);
  return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(unsigned* fault, unsigned long long timeout_ns,
                                    cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(fault, timeout_ns);
  return cudaGetLastError();
}

}  // namespace dgemm
