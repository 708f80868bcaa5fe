// tcgen05 (5th-generation tensor core) and cluster helpers for sm_103a, as
// inline PTX: shared-memory matrix and instruction descriptors, MMA issue
// and commit, TMEM allocation and loads, and the cluster primitives a CTA
// pair needs.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace dgemm {

// ------------------------------------------------------------ tcgen05 PTX

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor for kind::f16: FP32 accumulator, A and B of one
// type (0 = FP16, 1 = BF16), M = m, N = n; a_mn / b_mn = 1 when that
// operand is MN-major in shared memory (M or N contiguous), 0 when K-major.
__host__ __device__ constexpr uint32_t instr_desc(uint32_t ab_type, uint32_t m, uint32_t n,
                                                  uint32_t a_mn = 0, uint32_t b_mn = 1) {
  return (1u << 4)                 // D format: FP32
         | (ab_type << 7)          // A format
         | (ab_type << 10)         // B format
         | (a_mn << 15)            // A major
         | (b_mn << 16)            // B major
         | ((n >> 3) << 17)
         | ((m >> 4) << 24);
}

// Shared-memory descriptors of one 16-deep k-step, 128-byte swizzled, 8-row
// groups 1024 bytes apart:
//  * K-major (rows of 64 k, 128 bytes): +32 bytes per k-step within one
//    64-deep block (k16 = 0..3; a deeper stage keeps further blocks apart);
//  * MN-major (rows of 64 m or n, 128 bytes, one row per k; 64-wide blocks
//    block_bytes apart, i.e. 128 bytes x the stage depth): +16 rows = 2048
//    bytes per k-step over the whole stage depth, leading offset block_bytes.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int k16) {
  return smem_desc(base + k16 * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int k16,
                                                 uint32_t block_bytes = 8192) {
  return smem_desc(base + k16 * 2048, block_bytes, 1024);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when all tcgen05 operations this thread issued so
// far have completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 32 consecutive FP32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Waits for this thread's tcgen05.ld loads into r0 and r1.  tcgen05.ld writes
// its registers asynchronously, so the wait names them as read-write
// operands: no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r0)[32], uint32_t (&r1)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r0[0]), "+r"(r0[1]), "+r"(r0[2]), "+r"(r0[3]), "+r"(r0[4]), "+r"(r0[5]),
        "+r"(r0[6]), "+r"(r0[7]), "+r"(r0[8]), "+r"(r0[9]), "+r"(r0[10]), "+r"(r0[11]),
        "+r"(r0[12]), "+r"(r0[13]), "+r"(r0[14]), "+r"(r0[15]), "+r"(r0[16]), "+r"(r0[17]),
        "+r"(r0[18]), "+r"(r0[19]), "+r"(r0[20]), "+r"(r0[21]), "+r"(r0[22]), "+r"(r0[23]),
        "+r"(r0[24]), "+r"(r0[25]), "+r"(r0[26]), "+r"(r0[27]), "+r"(r0[28]), "+r"(r0[29]),
        "+r"(r0[30]), "+r"(r0[31])
      :
      : "memory");
  asm volatile(
      ""
      : "+r"(r1[0]), "+r"(r1[1]), "+r"(r1[2]), "+r"(r1[3]), "+r"(r1[4]), "+r"(r1[5]),
        "+r"(r1[6]), "+r"(r1[7]), "+r"(r1[8]), "+r"(r1[9]), "+r"(r1[10]), "+r"(r1[11]),
        "+r"(r1[12]), "+r"(r1[13]), "+r"(r1[14]), "+r"(r1[15]), "+r"(r1[16]), "+r"(r1[17]),
        "+r"(r1[18]), "+r"(r1[19]), "+r"(r1[20]), "+r"(r1[21]), "+r"(r1[22]), "+r"(r1[23]),
        "+r"(r1[24]), "+r"(r1[25]), "+r"(r1[26]), "+r"(r1[27]), "+r"(r1[28]), "+r"(r1[29]),
        "+r"(r1[30]), "+r"(r1[31])
      :
      : "memory");
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------------ epilogue scaling

template <typename T>
__device__ __forceinline__ float elem_to_f32(T v);
template <>
__device__ __forceinline__ float elem_to_f32<__half>(__half v) { return __half2float(v); }
template <>
__device__ __forceinline__ float elem_to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ float2 pair_to_f32(uint32_t bits);
template <>
__device__ __forceinline__ float2 pair_to_f32<__half>(uint32_t bits) {
  return __half22float2(*reinterpret_cast<const __half2*>(&bits));
}
template <>
__device__ __forceinline__ float2 pair_to_f32<__nv_bfloat16>(uint32_t bits) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bits));
}

// The old C of row `row`, columns col..col+63 (element type T, leading
// dimension ldc), as 8 groups of 8 raw elements; zero bits (the value 0)
// outside M x N.  16-byte loads where a group of 8 is in bounds.  Issued by
// the epilogue one chunk ahead of its use, and for a unit's first chunk
// before the wait for the accumulator, so that its latency is hidden.
template <typename T>
__device__ __forceinline__ void load_old_row64(uint4 (&raw)[8], const T* c_in, long long ldc,
                                               int M, int N, int row, int col) {
  const unsigned short* src =
      reinterpret_cast<const unsigned short*>(c_in) + (long long)row * ldc + col;
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    if (row < M && col + 8 * g + 8 <= N) {
      raw[g] = *reinterpret_cast<const uint4*>(src + 8 * g);
    } else {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c0 = col + 8 * g + 2 * e;
        const uint32_t lo = (row < M && c0 < N) ? src[8 * g + 2 * e] : 0u;
        const uint32_t hi = (row < M && c0 + 1 < N) ? src[8 * g + 2 * e + 1] : 0u;
        w[e] = lo | (hi << 16);
      }
      raw[g] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// v := alpha * v + beta * C_old on the 64 FP32 accumulator values (bits in
// r0[0..31], r1[0..31]) of one row; `old` (from load_old_row64) is read
// only when beta != 0.
template <typename T>
__device__ __forceinline__ void scale_row64(uint32_t (&r0)[32], uint32_t (&r1)[32], float alpha,
                                            float beta, const uint4 (&old)[8]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    r0[j] = __float_as_uint(alpha * __uint_as_float(r0[j]));
    r1[j] = __float_as_uint(alpha * __uint_as_float(r1[j]));
  }
  if (beta == 0.f) return;
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    uint32_t* dst = g < 4 ? &r0[g * 8] : &r1[(g - 4) * 8];
    const float2 a = pair_to_f32<T>(old[g].x), b = pair_to_f32<T>(old[g].y);
    const float2 c = pair_to_f32<T>(old[g].z), d = pair_to_f32<T>(old[g].w);
    const float o[8] = {a.x, a.y, b.x, b.y, c.x, c.y, d.x, d.y};
#pragma unroll
    for (int e = 0; e < 8; ++e)
      dst[e] = __float_as_uint(fmaf(beta, o[e], __uint_as_float(dst[e])));
  }
}

// The ragged tail of C, columns [n_tma, N) (fewer than 8; n_tma a multiple
// of 8), that the TMA store of a 64-column box leaves out: read back from
// this lane's staged row (128-byte swizzled, 16-byte chunk ch at
// (ch ^ (lane & 7)) * 16) and written with 2-byte stores.  `col` is the
// box's first global column (a multiple of 64); only the box holding
// column n_tma, and rows below M, write anything.
__device__ __forceinline__ void store_tail_row(const unsigned char* staged_row, int lane,
                                               void* c_out, long long ldc, int M, int N,
                                               int n_tma, int row, int col) {
  if (n_tma == N || n_tma < col || n_tma >= col + 64 || row >= M) return;
  const int ch = (n_tma - col) >> 3;
  const uint4 v = *reinterpret_cast<const uint4*>(staged_row + ((ch ^ (lane & 7)) << 4));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  unsigned short* dst = static_cast<unsigned short*>(c_out) + (long long)row * ldc + n_tma;
#pragma unroll
  for (int e = 0; e < 7; ++e)
    if (n_tma + e < N) dst[e] = (unsigned short)(w[e >> 1] >> (16 * (e & 1)));
}

// ------------------------------------------------------------ CTA pairs

// 2-CTA (cta_group::2) forms: one thread of the even CTA of a cluster pair
// issues an MMA of M = 256 whose A rows 0..127 and B columns [0, N/2) come
// from its own shared memory and A rows 128..255 and B columns [N/2, N)
// from the peer's, at the same offsets; each CTA's TMEM receives its own
// 128 rows of D.
__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once, when the pair's MMAs issued so far complete, on the mbarrier
// at shared offset `bar` of every CTA in `cta_mask`.
__device__ __forceinline__ void mma_commit_pair_multicast(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Arrive on an mbarrier given by its shared::cluster address (any CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// 2-D TMA load into this CTA's shared memory whose completion is counted on
// an mbarrier given by its shared::cluster address (the pair's even CTA).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* desc,
                                                 uint32_t cluster_bar, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(desc)), "r"(cluster_bar), "r"(x), "r"(y)
      : "memory");
}

// tma_load_2d_pair with an L2 cache-policy operand.
__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst, const CUtensorMap* desc,
                                                      uint32_t cluster_bar, int32_t x, int32_t y,
                                                      uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(desc)), "r"(cluster_bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// The pair load of operand kOperand (0 = A, 1 = B) under DENSE_GEMM_L2_HINT.
template <int kOperand>
__device__ __forceinline__ void tma_load_operand_pair(uint32_t dst, const CUtensorMap* desc,
                                                      uint32_t cluster_bar, int32_t x, int32_t y) {
#if DENSE_GEMM_L2_HINT == 0
  tma_load_2d_pair(dst, desc, cluster_bar, x, y);
#else
  tma_load_2d_pair_hint(dst, desc, cluster_bar, x, y,
                        l2_policy((DENSE_GEMM_L2_HINT == 1) == (kOperand == 0)));
#endif
}

}  // namespace dgemm
