// FP32 SIMT SGEMM for sm_103a: C = A . B, all row-major, FP32 FFMA with FP32
// accumulation (no TF32).
//
// Lineage on the pages, and what changed for GB300:
//  * Block tiling with a register-blocked outer product, 8 x 8 outputs per
//    thread and a 128 x 128 block tile ("[CUDA 优化实战] sgemm - 超越 cuBLAS",
//    section 2 and its resource-sizing analysis; "GEMM：从朴素实现到 shared memory
//    tiling 与寄存器分块", section 3; m.lqnn.cn SGEMM article, the v3 register
//    micro-tile).
//  * 16-byte fragment loads from shared memory (wingedge777 section 3 reads A
//    fragments as float4 after transposing A into shared memory).  Here A is
//    not transposed: TMA cannot transpose 4-byte elements, so A stays
//    K-contiguous and each LDS.128 returns four k-steps of one row.  The
//    instruction count per FFMA is the same (2 A + 2 B LDS.128 per 64 FFMA).
//  * An XOR-swizzled shared-memory layout that makes every fragment read
//    conflict-free (wingedge777 section 4's SWIZZLE_A idea; GB300 roadmap
//    m.nxbn.cn section 3.3).  The A tile uses the pattern TMA's 128-byte
//    swizzle writes: 16-byte chunk q of row m lives at chunk q ^ (m mod 8).
//    A warp's four row groups are interleaved (thread row tr owns rows
//    tr + 4i) so that its four distinct rows fall in four distinct chunks.
//  * Coalesced 16-byte C stores: each warp writes whole 128-byte row segments
//    (wingedge777 section 5's write-back re-mapping).
//  * A multi-stage pipeline (wingedge777 section 6 double buffer; m.lqnn.cn v4
//    cp.async double buffer; m.nxbn.cn section 3.1-3.2 three or four stages and
//    TMA).  Here: a 3-stage ring filled by TMA (one thread issues both tile
//    copies, completion on an mbarrier) or, when a base or leading dimension
//    is not 16-byte aligned, by 4-byte cp.async with zero fill completing on
//    the same mbarrier.  One __syncthreads per 32-deep k-tile releases a slot.
//  * Tile rasterisation in groups of 16 tile rows, so that CTAs running at
//    the same time share A rows and B columns in L2 (the grid shape of the
//    library kernel noted in wingedge777 section "ncu 报告").
#include "launch.h"
#include "ptx.cuh"

namespace dgemm {
namespace {

constexpr int BM = kSgemmBM;
constexpr int BN = kSgemmBN;
constexpr int BK = kSgemmBK;
constexpr int S = kSgemmStages;
constexpr int kAStageFloats = BM * BK;
constexpr int kBStageFloats = BK * BN;
constexpr uint32_t kStageBytes = (kAStageFloats + kBStageFloats) * 4;

static_assert(BK == 32, "A tile rows must be 128 bytes for the 128-byte swizzle");
static_assert(kSgemmThreads == 256, "thread mapping below assumes 8 warps");

// Offset (in floats) of A element (m, k) inside one A stage: rows of 32
// floats, 16-byte chunk index XOR-ed with the row index mod 8.
__host__ __device__ constexpr int a_tile_offset(int m, int k) {
  return m * BK + ((((k >> 2) ^ (m & 7))) << 2) + (k & 3);
}

// Offset (in floats) of B element (k, n) inside one B stage: plain rows of
// 128 floats; a warp always reads 8 consecutive 16-byte chunks of one row.
__host__ __device__ constexpr int b_tile_offset(int k, int n) { return k * BN + n; }

__device__ __forceinline__ float4 lds128(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

template <bool kTma>
__global__ void __launch_bounds__(kSgemmThreads, 2)
    sgemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const SgemmParams p) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ int s_abort;
  const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
  float* sA = reinterpret_cast<float*>(base);
  float* sB = sA + S * kAStageFloats;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + S * kBStageFloats);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  // Grouped rasterisation: consecutive CTAs walk down a group of
  // kSgemmGroupM tile rows before moving one tile column to the right.
  int tm, tn;
  {
    const int t = blockIdx.x;
    const int per_group = kSgemmGroupM * p.tiles_n;
    const int group = t / per_group;
    const int first_m = group * kSgemmGroupM;
    const int gsize = min(p.tiles_m - first_m, kSgemmGroupM);
    const int r = t - group * per_group;
    tm = first_m + r % gsize;
    tn = r / gsize;
  }
  const int m0 = tm * BM;
  const int n0 = tn * BN;
  const int nk = (p.K + BK - 1) / BK;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), kTma ? 1u : kSgemmThreads);
    s_abort = 0;
    fence_mbar_init();
    if constexpr (kTma) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
    }
  }
  __syncthreads();

  // Stage k-tile kt into ring slot s.
  auto issue = [&](int kt, int s) {
    const int k0 = kt * BK;
    const uint32_t bar = smem_u32(&full[s]);
    if constexpr (kTma) {
      if (tid == 0) {
        mbar_arrive_expect_tx(bar, kStageBytes);
        tma_load_2d(smem_u32(sA + s * kAStageFloats), &tmA, bar, k0, m0);
        tma_load_2d(smem_u32(sB + s * kBStageFloats), &tmB, bar, n0, k0);
      }
    } else {
      // A: a warp copies one 32-float row segment (k contiguous in memory).
      const uint32_t a_dst = smem_u32(sA + s * kAStageFloats);
      const int ka = tid & 31;
      const int gk = k0 + ka;
#pragma unroll
      for (int j = 0; j < BM / 8; ++j) {
        const int m = (tid >> 5) + 8 * j;
        const int gm = m0 + m;
        const bool v = (gm < p.M) && (gk < p.K);
        const float* src = v ? p.A + (long long)gm * p.lda + gk : p.A;
        cp_async_4(a_dst + 4u * a_tile_offset(m, ka), src, v);
      }
      // B: 128 threads copy one 128-float row segment (n contiguous).
      const uint32_t b_dst = smem_u32(sB + s * kBStageFloats);
      const int nb = tid & (BN - 1);
      const int gn = n0 + nb;
#pragma unroll
      for (int j = 0; j < BK / 2; ++j) {
        const int k = (tid >> 7) + 2 * j;
        const int gk2 = k0 + k;
        const bool v = (gk2 < p.K) && (gn < p.N);
        const float* src = v ? p.B + (long long)gk2 * p.ldb + gn : p.B;
        cp_async_4(b_dst + 4u * b_tile_offset(k, nb), src, v);
      }
      cp_async_mbar_arrive_noinc(bar);
    }
  };

  const int pre = nk < S ? nk : S;
  for (int kt = 0; kt < pre; ++kt) issue(kt, kt);

  // Thread -> output mapping.  Warp (warp_m, warp_n) owns a 32 x 64 block;
  // lane (tr, tc) owns rows tr + 4i (i < 8) and columns tc*4 + {0..3} and
  // 32 + tc*4 + {0..3} of it.
  const int warp_m = warp >> 1;
  const int warp_n = warp & 1;
  const int tr = lane >> 3;
  const int tc = lane & 7;
  const int a_row0 = warp_m * 32 + tr;            // row for i = 0
  const int b_col0 = warp_n * 64 + tc * 4;

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  int kt = 0;
  for (; kt < nk; ++kt) {
    const int s = kt % S;
    const bool ok = mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((kt / S) & 1), p.timeout_ns,
                                      &s_abort);
    if (!ok) {
      s_abort = 1;
    } else {
      const float* As = sA + s * kAStageFloats;
      const float* Bs = sB + s * kBStageFloats + b_col0;
      // Row (a_row0 + 4i) mod 8 = tr + 4 (i mod 2): its chunk for k-quad kq is
      // kq ^ tr ^ 4(i mod 2).  Four base pointers cover (kq mod 4) ^ tr.
      const float* a_base[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) a_base[q] = As + a_row0 * BK + (((q ^ tr) & 3) << 2);
#pragma unroll
      for (int kq = 0; kq < BK / 4; ++kq) {
        float4 a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          a[i] = lds128(a_base[kq & 3] + 4 * i * BK + (((kq & 4) ^ ((i & 1) << 2)) << 2));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float* brow = Bs + (kq * 4 + kk) * BN;
          const float4 b0 = lds128(brow);
          const float4 b1 = lds128(brow + 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float av = (&a[i].x)[kk];
            acc[i][0] = fmaf(av, b0.x, acc[i][0]);
            acc[i][1] = fmaf(av, b0.y, acc[i][1]);
            acc[i][2] = fmaf(av, b0.z, acc[i][2]);
            acc[i][3] = fmaf(av, b0.w, acc[i][3]);
            acc[i][4] = fmaf(av, b1.x, acc[i][4]);
            acc[i][5] = fmaf(av, b1.y, acc[i][5]);
            acc[i][6] = fmaf(av, b1.z, acc[i][6]);
            acc[i][7] = fmaf(av, b1.w, acc[i][7]);
          }
        }
      }
    }
    // Every thread is done with slot s (or some thread gave up).
    if (__syncthreads_or(!ok)) break;
    if (kt + S < nk) issue(kt + S, s);
  }

  if (kt < nk) {
    // A wait gave up: record it, let this CTA's own copies land, and leave
    // without writing C.
    if (tid == 0) raise_fault(p.fault, kFaultSgemmFullWait);
    if constexpr (kTma) {
      if (tid == 0) {
        const int issued = (kt + S < nk) ? kt + S : nk;
        for (int t = kt; t < issued; ++t) {
          if (!mbar_wait_bounded(smem_u32(&full[t % S]), (uint32_t)((t / S) & 1), p.timeout_ns,
                                 nullptr)) {
            raise_fault(p.fault, kFaultDrainWait);
            break;
          }
        }
      }
    } else {
      cp_async_wait_all();
    }
    __syncthreads();
    return;
  }

  // Epilogue: each store instruction of a warp covers four full 128-byte row
  // segments of C.
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gm = m0 + a_row0 + 4 * i;
    if (gm >= p.M) continue;
    float* crow = p.C + (long long)gm * p.ldc;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int gn = n0 + b_col0 + 32 * h;
      const float v0 = acc[i][4 * h + 0], v1 = acc[i][4 * h + 1];
      const float v2 = acc[i][4 * h + 2], v3 = acc[i][4 * h + 3];
      if (p.c_vec4 && gn + 3 < p.N) {
        *reinterpret_cast<float4*>(crow + gn) = make_float4(v0, v1, v2, v3);
      } else {
        if (gn + 0 < p.N) crow[gn + 0] = v0;
        if (gn + 1 < p.N) crow[gn + 1] = v1;
        if (gn + 2 < p.N) crow[gn + 2] = v2;
        if (gn + 3 < p.N) crow[gn + 3] = v3;
      }
    }
  }
}

}  // namespace

cudaError_t launch_sgemm(const SgemmParams& p, bool use_tma, const CUtensorMap* tmA,
                         const CUtensorMap* tmB, cudaStream_t stream) {
  // The attribute is per function; setting it on every call is cheap and
  // keeps this correct for every device of the process.
  cudaError_t e;
  const dim3 grid((unsigned)(p.tiles_m * p.tiles_n));
  if (use_tma) {
    e = cudaFuncSetAttribute(sgemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSgemmSmemBytes);
    if (e != cudaSuccess) return e;
    sgemm_kernel<true><<<grid, kSgemmThreads, kSgemmSmemBytes, stream>>>(*tmA, *tmB, p);
  } else {
    e = cudaFuncSetAttribute(sgemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSgemmSmemBytes);
    if (e != cudaSuccess) return e;
    CUtensorMap none{};
    sgemm_kernel<false><<<grid, kSgemmThreads, kSgemmSmemBytes, stream>>>(none, none, p);
  }
  return cudaGetLastError();
}

// Host-visible copy of the A / B stage layouts, for layout checks on the CPU.
int sgemm_smem_offset(int which, int r, int c) {
  return which == 0 ? a_tile_offset(r, c) : b_tile_offset(r, c);
}

}  // namespace dgemm
