// Internal interface between the C-ABI dispatcher (api.cu) and the kernel
// translation units.  Not installed; callers use include/dense_gemm.h.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

namespace dgemm {

// ---------------------------------------------------------------- FP32 SIMT

// Block tile 128 x 128 x 32, 256 threads (8 warps of 32 x 64), 8 x 8 outputs
// per thread, a 3-stage shared-memory ring, two CTAs per SM.
constexpr int kSgemmBM = 128;
constexpr int kSgemmBN = 128;
constexpr int kSgemmBK = 32;
constexpr int kSgemmStages = 3;
constexpr int kSgemmThreads = 256;
constexpr int kSgemmGroupM = 16;   // tile rows per rasterisation group (L2 reuse)
constexpr int kSgemmSmemBytes =
    kSgemmStages * (kSgemmBM * kSgemmBK + kSgemmBK * kSgemmBN) * 4 + 1024 /*align*/ + 64;

struct SgemmParams {
  int M, N, K;
  const float* A;
  long long lda;
  const float* B;
  long long ldb;
  float* C;
  long long ldc;
  int tiles_m, tiles_n;
  int c_vec4;        // C rows may be written with 16-byte stores
  unsigned* fault;   // device fault word
  unsigned long long timeout_ns;
};

// use_tma: A and B are staged by TMA (16-byte aligned bases and strides);
// otherwise by 4-byte cp.async with zero fill.  Returns the launch error.
cudaError_t launch_sgemm(const SgemmParams& p, bool use_tma, const CUtensorMap* tmA,
                         const CUtensorMap* tmB, cudaStream_t stream);

// Element offset of (row, col) inside one stage of the FP32 A tile
// (which = 0) or B tile (which = 1); host copy of the device layout.
int sgemm_smem_offset(int which, int r, int c);

// ---------------------------------------------------------------- FP16/BF16 tcgen05

// Output tile 128 x 256 per CTA (one tcgen05.mma M=128, N=256 accumulator,
// double-buffered in tensor memory), k-tile 64, 4-stage TMA ring, persistent
// grid of at most one CTA per SM.
constexpr int kTcBM = 128;
constexpr int kTcBN = 256;
constexpr int kTcBK = 64;
constexpr int kTcStages = 4;
constexpr int kTcThreads = 192;          // producer warp, MMA warp, 4 epilogue warps
constexpr int kTcGroupM = 8;             // tile rows per rasterisation group
constexpr int kTcEpiCols = 64;           // columns per epilogue store box
constexpr int kTcSmemBytes =
    kTcStages * (kTcBM * kTcBK + kTcBK * kTcBN) * 2   // A and B ring
    + 4 * 2 * 32 * kTcEpiCols * 2                     // 4 warps x 2 buffers x 32 x 64 x 2 B
    + 1024 /*align*/ + 256 /*barriers*/;

struct TcParams {
  int M, N, K;
  int tiles_m, tiles_n;
  unsigned* fault;
  unsigned long long timeout_ns;
};

// dtype: 1 = FP16, 2 = BF16.  tmA: A as {K, M} with 64 x 128 boxes;
// tmB: B as {N, K} with 64 x 64 boxes; tmC: C as {N, M} with 64 x 32 boxes;
// all 128-byte swizzled.  grid = number of persistent CTAs.
cudaError_t launch_gemm_tc(int dtype, const TcParams& p, const CUtensorMap* tmA,
                           const CUtensorMap* tmB, const CUtensorMap* tmC, int grid,
                           cudaStream_t stream);

// ---------------------------------------------------------------- zero fill

// C[i][j] = 0 for i < M, j < N (row-major, leading dimension ldc, element
// size elem_bytes = 2 or 4): the K == 0 product.
cudaError_t launch_zero_fill(void* C, int M, int N, long long ldc, int elem_bytes,
                             cudaStream_t stream);

// ---------------------------------------------------------------- self test

// Waits on an mbarrier that nothing completes, with a `timeout_ns` bound; the
// wait gives up, records kFaultSelftestWait and the kernel returns.
cudaError_t launch_selftest_timeout(unsigned* fault, unsigned long long timeout_ns,
                                    cudaStream_t stream);

}  // namespace dgemm
