// Small kernels around the GEMM path: the K == 0 / alpha == 0 product
// (C := beta * C), the split-K slice reduction, the FP32 operand transpose
// that packs a transposed operand into row-major scratch, the re-pitch of
// an operand with unaligned rows, and the self-tests of the bounded waits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "launch.h"
#include "ptx.cuh"

namespace dgemm {
namespace {

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

// One thread waits for a global flag that nothing sets (the K-split
// hand-over's wait); it gives up after timeout_ns and records
// kFaultTcPartialWait.
__device__ unsigned g_selftest_flag;   // stays 0
__global__ void selftest_flag_kernel(unsigned* fault, unsigned long long timeout_ns) {
  if (threadIdx.x != 0) return;
  if (!flag_wait_equal(&g_selftest_flag, 1u, timeout_ns, nullptr))
    raise_fault(fault, kFaultTcPartialWait);
}

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Sums the split-K slices of each output element in slice order and rounds
// once.  Consecutive threads take consecutive columns (coalesced reads of
// every slice and coalesced writes of C).
template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T>
__global__ void splitk_reduce_kernel(const float* __restrict__ ws, int slices, int M, int N,
                                     long long ldw, T* __restrict__ C, long long ldc, float alpha,
                                     float beta, int c_trans) {
  const long long total = (long long)M * N;
  const long long slice_stride = (long long)M * ldw;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long i = idx / N;
    const long long j = idx - i * N;
    const float* src = ws + i * ldw + j;
    float acc = __ldg(src);
    for (int s = 1; s < slices; ++s) acc += __ldg(src + s * slice_stride);
    float v = alpha * acc;
    T* c = C + (c_trans ? j * ldc + i : i * ldc + j);
    if (beta != 0.f) v = fmaf(beta, to_f32<T>(*c), v);
    *c = from_f32<T>(v);
  }
}

template <typename T>
__global__ void scale_c_kernel(T* C, int M, int N, long long ldc, float beta) {
  const long long total = (long long)M * N;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long i = idx / N;
    const long long j = idx - i * N;
    T* c = C + i * ldc + j;
    *c = beta == 0.f ? T(0) : from_f32<T>(beta * to_f32<T>(*c));
  }
}

// D (cols x rows, row pitch ldd) := transpose of S (rows x cols, row pitch
// lds), through 64 x 64 tiles in shared memory so that both the reads of S
// and the writes of D are whole 128-byte row segments.  Each thread first
// issues its 16 loads, then stores them; the tile's row pitch of 65 words
// keeps both the row-wise writes and the column-wise reads of shared
// memory free of bank conflicts.  HBM-bound: every element is read once
// and written once.
constexpr int kTrTile = 64;
constexpr int kTrThreads = 256;

__global__ void __launch_bounds__(kTrThreads)
    transpose_f32_kernel(const float* __restrict__ S, long long rows, long long cols,
                         long long lds, float* __restrict__ D, long long ldd) {
  __shared__ float tile[kTrTile][kTrTile + 1];
  constexpr int kPer = kTrTile * kTrTile / kTrThreads;   // 16
  constexpr int kRowsPerPass = kTrThreads / kTrTile;     // 4
  const int t = threadIdx.x;
  const int tc = t % kTrTile, tr = t / kTrTile;
  const long long tiles_c = (cols + kTrTile - 1) / kTrTile;
  const long long tiles = (rows + kTrTile - 1) / kTrTile * tiles_c;
  for (long long tile_id = blockIdx.x; tile_id < tiles; tile_id += gridDim.x) {
    const long long r0 = tile_id / tiles_c * kTrTile;
    const long long c0 = tile_id % tiles_c * kTrTile;
    float v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const long long r = r0 + i * kRowsPerPass + tr, c = c0 + tc;
      v[i] = (r < rows && c < cols) ? __ldcs(S + r * lds + c) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) tile[i * kRowsPerPass + tr][tc] = v[i];
    __syncthreads();
    // Row c of D holds column c of S: lane tc writes D[c0 + c][r0 + tc].
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const long long c = c0 + i * kRowsPerPass + tr, r = r0 + tc;
      if (c < cols && r < rows) D[c * ldd + r] = tile[tc][i * kRowsPerPass + tr];
    }
    __syncthreads();
  }
}

// Copies each job's S (lds) into D (ldd, 16-byte rows): item i of the
// grid-stride loop over both jobs' quads takes the 4 columns 4q .. 4q + 3
// of one row, reads them as scalars (a warp reads 512 contiguous bytes) and
// writes one 16-byte store; columns from cols on are written as zeros.
__global__ void __launch_bounds__(256)
    repitch_f32_kernel(RepitchJob j0, RepitchJob j1, int njobs) {
  const long long q0 = j0.rows * (j0.ldd / 4);
  const long long total = q0 + (njobs > 1 ? j1.rows * (j1.ldd / 4) : 0);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const bool second = i >= q0;
    const RepitchJob& j = second ? j1 : j0;
    const long long k = second ? i - q0 : i;
    const long long quads = j.ldd / 4;
    const long long r = k / quads, c = (k - r * quads) * 4;
    const float* src = j.S + r * j.lds + c;
    float4 v;
    v.x = c < j.cols ? __ldcs(src) : 0.f;
    v.y = c + 1 < j.cols ? __ldcs(src + 1) : 0.f;
    v.z = c + 2 < j.cols ? __ldcs(src + 2) : 0.f;
    v.w = c + 3 < j.cols ? __ldcs(src + 3) : 0.f;
    *reinterpret_cast<float4*>(j.D + r * j.ldd + c) = v;
  }
}

}  // namespace

cudaError_t launch_repitch_f32(const RepitchJob* jobs, int njobs, int sms, cudaStream_t stream) {
  if (njobs < 1 || njobs > 2) return cudaErrorInvalidValue;
  long long total = 0;
  for (int i = 0; i < njobs; ++i) total += jobs[i].rows * (jobs[i].ldd / 4);
  long long blocks = (long long)(sms > 0 ? sms : 1) * 8;
  if (blocks * 256 > total) blocks = (total + 255) / 256;
  if (blocks < 1) blocks = 1;
  repitch_f32_kernel<<<(unsigned)blocks, 256, 0, stream>>>(jobs[0], jobs[njobs - 1], njobs);
  return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const float* ws, int slices, int M, int N, long long ldw,
                                 void* C, long long ldc, int elem, float alpha, float beta,
                                 cudaStream_t stream, int c_trans) {
  const long long total = (long long)M * N;
  long long blocks = (total + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  if (elem == 0)
    splitk_reduce_kernel<float><<<(unsigned)blocks, 256, 0, stream>>>(
        ws, slices, M, N, ldw, static_cast<float*>(C), ldc, alpha, beta, c_trans);
  else if (elem == 1)
    splitk_reduce_kernel<__half><<<(unsigned)blocks, 256, 0, stream>>>(
        ws, slices, M, N, ldw, static_cast<__half*>(C), ldc, alpha, beta, c_trans);
  else
    splitk_reduce_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, stream>>>(
        ws, slices, M, N, ldw, static_cast<__nv_bfloat16*>(C), ldc, alpha, beta, c_trans);
  return cudaGetLastError();
}

cudaError_t launch_scale_c(void* C, int M, int N, long long ldc, int elem, float beta,
                           cudaStream_t stream) {
  const long long total = (long long)M * N;
  long long blocks = (total + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  if (elem == 0)
    scale_c_kernel<float><<<(unsigned)blocks, 256, 0, stream>>>(static_cast<float*>(C), M, N, ldc,
                                                                beta);
  else if (elem == 1)
    scale_c_kernel<__half><<<(unsigned)blocks, 256, 0, stream>>>(static_cast<__half*>(C), M, N,
                                                                 ldc, beta);
  else
    scale_c_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<__nv_bfloat16*>(C), M, N, ldc, beta);
  return cudaGetLastError();
}

cudaError_t launch_transpose_f32(const float* S, long long rows, long long cols, long long lds,
                                 float* D, long long ldd, int sms, cudaStream_t stream) {
  const long long tiles = (rows + kTrTile - 1) / kTrTile * ((cols + kTrTile - 1) / kTrTile);
  // 8 resident CTAs of 256 threads per SM; the loop strides over tiles.
  long long blocks = (long long)(sms > 0 ? sms : 1) * 8 * 4;
  if (blocks > tiles) blocks = tiles;
  if (blocks < 1) blocks = 1;
  transpose_f32_kernel<<<(unsigned)blocks, kTrThreads, 0, stream>>>(S, rows, cols, lds, D, ldd);
  return cudaGetLastError();
}

cudaError_t launch_selftest_flag_timeout(unsigned* fault, unsigned long long timeout_ns,
                                         cudaStream_t stream) {
  selftest_flag_kernel<<<1, 32, 0, stream>>>(fault, timeout_ns);
  return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(unsigned* fault, unsigned long long timeout_ns,
                                    cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(fault, timeout_ns);
  return cudaGetLastError();
}

}  // namespace dgemm
