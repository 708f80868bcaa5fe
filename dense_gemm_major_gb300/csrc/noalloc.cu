// gemm_f32_noalloc: the FP32 GEMM for callers that cannot allocate device
// memory (see include/dense_gemm.h).  It runs as gemm_f32 with operand
// copies turned off (an unaligned operand is staged by cp.async, never
// re-pitched into scratch), and split-K partial tiles and stream-K
// hand-over flags kept in the fixed arrays below instead of library-
// allocated ones.
#include <atomic>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "dense_gemm.h"
#include "launch.h"

namespace {

// The scratch: 16 MiB of FP32 split-K partials, one copy per device that
// loads this code, kept until the process exits.  Host code must not use
// the symbol as a pointer; it only names the array for cudaGetSymbolAddress.
constexpr size_t kScratchBytes = 16u << 20;
static __device__ __align__(256) float g_noalloc_scratch[kScratchBytes / sizeof(float)];
// The stream-K hand-over flags of the calls that are not split-K (two words
// per CTA boundary; zero at load, then only ever set to a call's epoch).
constexpr long long kFlagWords = 8192;
static __device__ unsigned g_noalloc_flags[kFlagWords];

constexpr int kMaxDevices = 64;

struct ScratchDevice {
  bool ready = false;
  float* scratch = nullptr;   // device address of g_noalloc_scratch on this device
  unsigned* flags = nullptr;  // device address of g_noalloc_flags
  std::atomic<unsigned> epoch{0};
};

std::mutex g_mu;
ScratchDevice g_dev[kMaxDevices];

// Once per device, with that device current: the arrays' device addresses.
gemm_status_t scratch_device(ScratchDevice** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GEMM_ERR_UNSUPPORTED_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchDevice& d = g_dev[dev];
  if (!d.ready) {
    void* ptr = nullptr;
    void* fptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess ||
        cudaGetSymbolAddress(&fptr, g_noalloc_flags) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    d.scratch = static_cast<float*>(ptr);
    d.flags = static_cast<unsigned*>(fptr);
    d.ready = true;
  }
  *out = &d;
  return GEMM_OK;
}

}  // namespace

extern "C" gemm_status_t gemm_f32_noalloc(int M, int N, int K, const float* A, int lda,
                                          const float* B, int ldb, float* C, int ldc,
                                          cudaStream_t stream) {
  // Argument checks first (no device needed), as for gemm_f32.
  gemm_plan_t plan;
  gemm_status_t st = gemm_plan(0, M, N, K, A, lda, B, ldb, C, ldc, 1, &plan);
  if (st != GEMM_OK || plan.path == GEMM_PATH_NOOP) return st;
  ScratchDevice* dev = nullptr;
  st = scratch_device(&dev);
  if (st != GEMM_OK) return st;
  unsigned epoch = ++dev->epoch;
  if (epoch == 0) epoch = ++dev->epoch;
  const dgemm::FixedScratch scratch{dev->flags, kFlagWords, epoch, dev->scratch,
                                    (long long)kScratchBytes};
  return dgemm::run_f32_no_copy(M, N, K, A, lda, B, ldb, C, ldc, stream, scratch);
}
