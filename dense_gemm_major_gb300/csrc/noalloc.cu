// gemm_f32_noalloc: the FP32 GEMM for callers that cannot allocate device
// memory (see include/dense_gemm.h).  Split-K problems keep their FP32
// partial tiles in the fixed array below instead of a library-allocated
// workspace; everything else runs as gemm_f32 with operand copies turned
// off (an unaligned operand is staged by cp.async, never re-pitched into
// scratch) and the stream-K hand-over flags taken from a fixed array too.
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
  int sms = 0;
  std::atomic<unsigned> epoch{0};
};

std::mutex g_mu;
ScratchDevice g_dev[kMaxDevices];

// Once per device, with that device current: the array's device address and
// the SM count that plans the split.
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
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0) {
      cudaGetLastError();
      return GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    d.scratch = static_cast<float*>(ptr);
    d.flags = static_cast<unsigned*>(fptr);
    d.sms = sms;
    d.ready = true;
  }
  *out = &d;
  return GEMM_OK;
}

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace

extern "C" gemm_status_t gemm_f32_noalloc(int M, int N, int K, const float* A, int lda,
                                          const float* B, int ldb, float* C, int ldc,
                                          cudaStream_t stream) {
  // Argument checks first (no device needed), as for gemm_f32.
  gemm_plan_t plan;
  gemm_status_t st = dgemm::plan_f32_no_copy(M, N, K, A, lda, B, ldb, C, ldc, 1, &plan);
  if (st != GEMM_OK || plan.path == GEMM_PATH_NOOP) return st;
  ScratchDevice* dev = nullptr;
  st = scratch_device(&dev);
  if (st != GEMM_OK) return st;
  unsigned* fault = dgemm::current_fault_word();
  if (fault == nullptr) return GEMM_ERR_UNSUPPORTED_DEVICE;
  st = dgemm::plan_f32_no_copy(M, N, K, A, lda, B, ldb, C, ldc, dev->sms, &plan);
  if (st != GEMM_OK) return st;
  if (plan.splitk_slices <= 1) {
    unsigned e = ++dev->epoch;
    if (e == 0) e = ++dev->epoch;
    const dgemm::FixedFlags flags{dev->flags, kFlagWords, e};
    return dgemm::run_f32_no_copy(M, N, K, A, lda, B, ldb, C, ldc, stream, flags);
  }
  if (plan.workspace_bytes > (long long)kScratchBytes) return GEMM_ERR_SCRATCH_LIMIT;

  // Split-K with the static scratch: the narrow SIMT tile, tiles staged by
  // 4-byte cp.async (no tensor maps needed), then the slice reduction.
  dgemm::SgemmParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.A = A;
  p.lda = lda;
  p.B = B;
  p.ldb = ldb;
  p.C = C;
  p.ldc = ldc;
  p.tiles_m = ceil_div(M, dgemm::kSgemmBM);
  p.tiles_n = ceil_div(N, dgemm::sgemm_bn(8));
  p.grid = plan.ctas;
  p.split_tiles = 0;
  p.slices = plan.splitk_slices;
  p.ws = dev->scratch;
  p.ldw = ((long long)N + 3) / 4 * 4;
  p.alpha = 1.f;
  p.beta = 0.f;
  p.c_vec4 = 0;
  p.fault = fault;
  p.timeout_ns = dgemm::wait_bound_ns();
  cudaError_t e = dgemm::launch_sgemm(p, 8, /*use_tma=*/false, nullptr, nullptr, stream);
  if (e == cudaSuccess)
    e = dgemm::launch_splitk_reduce(p.ws, p.slices, M, N, p.ldw, C, ldc, 0, 1.f, 0.f, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}
