// FP32 SIMT SGEMM for sm_103a: C = A . B, all row-major, FP32 FFMA with FP32
// accumulation (no TF32).
//
// Lineage on the pages, and what changed for GB300:
//  * Block tiling with a register-blocked outer product, 8 x 8 outputs per
//    thread and a 128 x 128 block tile ("[CUDA 优化实战] sgemm - 超越 cuBLAS",
//    section 2 and its resource-sizing analysis; "GEMM：从朴素实现到 shared memory
//    tiling 与寄存器分块", section 3; m.lqnn.cn SGEMM article, the v3 register
//    micro-tile).  A wide configuration (8 x 16 per thread, 128 x 256 block
//    tile, one CTA per SM) serves grids of one to two narrow waves.
//  * Vector fragment loads from shared memory (wingedge777 section 3 reads A
//    fragments as float4 after transposing A into shared memory).  Here A is
//    not transposed: TMA cannot transpose 4-byte elements, so A stays
//    K-contiguous and one LDS.64 returns two k-steps of one row; B fragments
//    are LDS.128.  Measured on sm_103a with a shared-load probe: a wavefront
//    delivers one distinct 16-byte chunk to each group of 4 consecutive
//    lanes (broadcast within the group is free) and a 16-byte load costs at
//    least 2 wavefronts.  Each 4-lane group is therefore a 2 x 2 block of the
//    warp's 4 x 8 lane grid, so every fragment load costs the minimum, 8
//    bytes per lane per wavefront (0.125 wavefronts per FFMA at 8 x 8 outputs
//    per thread).
//  * An XOR-swizzled shared-memory layout that makes every fragment read
//    conflict-free (wingedge777 section 4's SWIZZLE_A idea; GB300 roadmap
//    m.nxbn.cn section 3.3).  The A tile uses the pattern TMA's 128-byte
//    swizzle writes: 16-byte chunk q of row m lives at chunk q ^ (m mod 8).
//    A warp's four row groups are interleaved (thread row tr owns rows
//    tr + 4i) so that its four distinct rows fall in four distinct chunks.
//  * Coalesced 16-byte C stores: each warp writes whole 128-byte row segments
//    (wingedge777 section 5's write-back re-mapping).
//  * The outer product is issued as packed fma.rn.f32x2 (two FP32 FMAs per
//    lane per instruction, each rounded like fmaf): scalar FFMA would need
//    every issue slot of an SM sub-partition to reach the FFMA peak.
//  * A multi-stage pipeline (wingedge777 section 6 double buffer; m.lqnn.cn v4
//    cp.async double buffer; m.nxbn.cn section 3.1-3.2 three or four stages and
//    TMA).  Here: a 3-, 4- or 6-stage ring filled by TMA (one thread issues both
//    tile copies, completion on an mbarrier) or, when a base or leading
//    dimension is not 16-byte aligned, by 4-byte cp.async with zero fill
//    completing on the same mbarrier.  One __syncthreads per S - 1 32-deep
//    k-tiles releases S - 1 slots (three of the wide tile's four; five of
//    six, or two of three, for the narrow tile at one or two CTAs per SM).
//  * Hybrid stream-K tile scheduling (see the unit loop below) instead of one
//    tile per CTA: full waves of whole tiles, then an equal share of the
//    remaining (tile, k-tile) iterations per CTA.
//  * Operands stored transposed (A as K x M, B as N x K: the column-major B
//    of the m.lqnn.cn article, section 3.1) are transposed while they are
//    staged: 4-byte cp.async scatters each element to its place in the same
//    shared-memory tiles, so the main loop is the same.  The lanes of one
//    copy instruction are chosen so that both sides are efficient: a
//    transposed A copy covers 8 m x 4 k (four 32-byte sectors in memory, 32
//    distinct banks in the swizzled A tile); a transposed B copy covers 4 n
//    x 8 k spaced by 4 (four 128-byte rows in memory, which the four copies
//    of a k-quad share in L1), and the transposed-B tile XORs its 16-byte
//    chunk index with k / 4 so that those 8 k land in 8 distinct chunks.
//  * Tile rasterisation in groups of 16 tile rows, so that CTAs running at
//    the same time share A rows and B columns in L2 (the grid shape of the
//    library kernel noted in wingedge777 section "ncu 报告").
#pragma once

#include "launch.h"
#include "ptx.cuh"

namespace dgemm {
namespace {

constexpr int BM = kSgemmBM;
constexpr int BK = kSgemmBK;
constexpr int kAStageFloats = BM * BK;

static_assert(BK == 32, "A tile rows must be 128 bytes for the 128-byte swizzle");
static_assert(kSgemmThreads == 256, "thread mapping below assumes 8 warps");

// Offset (in floats) of A element (m, k) inside one A stage: rows of 32
// floats, 16-byte chunk index XOR-ed with the row index mod 8.
__host__ __device__ constexpr int a_tile_offset(int m, int k) {
  return m * BK + ((((k >> 2) ^ (m & 7))) << 2) + (k & 3);
}

// Offset (in floats) of B element (k, n) inside one B stage of width BN:
// plain rows; a quarter warp always reads 8 consecutive 16-byte chunks of
// one row.
__host__ __device__ constexpr int b_tile_offset(int bn, int k, int n) { return k * bn + n; }

// The B stage of a transposed B: row k's 16-byte chunk c is stored at chunk
// c ^ ((k / 4) mod 8).  A quarter warp still reads 8 distinct chunks of one
// 128-byte segment of a row; the 8 k = 4l + kk (l < 8) of one transposing
// copy land in 8 distinct chunks.
__host__ __device__ constexpr int bt_tile_offset(int bn, int k, int n) {
  return k * bn + ((((n >> 2) ^ ((k >> 2) & 7))) << 2) + (n & 3);
}

// 16 bytes of shared memory as two packed float pairs (one LDS.128).
__device__ __forceinline__ ulonglong2 lds128_pairs(const float* p) {
  return *reinterpret_cast<const ulonglong2*>(p);
}

__device__ __forceinline__ unsigned long long pack_pair(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ float2 unpack_pair(unsigned long long v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}

// d.lo += a.lo * b.lo and d.hi += a.hi * b.hi, each one correctly rounded
// FMA (the same result as fmaf), issued as one packed instruction: half the
// issue slots of two scalar FFMA.
__device__ __forceinline__ void ffma2(unsigned long long& d, unsigned long long a,
                                      unsigned long long b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

// Offset of the kernel's output element (r, c) in C: row-major, or
// transposed when the product is computed as C^T (p.c_trans).
__host__ __device__ __forceinline__ long long c_index(const SgemmParams& p, int r, int c) {
  return p.c_trans ? (long long)c * p.ldc + r : (long long)r * p.ldc + c;
}
template <bool kCT>
__device__ __forceinline__ long long kc_index(const SgemmParams& p, int r, int c) {
  return kCT ? (long long)c * p.ldc + r : (long long)r * p.ldc + c;
}

// 4 x 4 transpose among the four lanes of a warp that share tc (their tr
// sits in lane bits 1 and 4): before, slot s of lane t holds row 4s + t of
// a 16-row block; after, slot r of lane t holds row 4t + r.  Two butterfly
// steps, each swapping one bit of the lane's tr with the same bit of the
// slot index.  All 32 lanes must take part.
__device__ __forceinline__ void transpose4_lanes(float (&x)[4], int tr) {
  {
    const bool t0 = (tr & 1) != 0;
    float a = t0 ? x[0] : x[1];
    float b = t0 ? x[2] : x[3];
    a = __shfl_xor_sync(0xffffffffu, a, 2);
    b = __shfl_xor_sync(0xffffffffu, b, 2);
    if (t0) {
      x[0] = a;
      x[2] = b;
    } else {
      x[1] = a;
      x[3] = b;
    }
  }
  {
    const bool t1 = (tr & 2) != 0;
    float a = t1 ? x[0] : x[2];
    float b = t1 ? x[1] : x[3];
    a = __shfl_xor_sync(0xffffffffu, a, 16);
    b = __shfl_xor_sync(0xffffffffu, b, 16);
    if (t1) {
      x[0] = a;
      x[1] = b;
    } else {
      x[2] = a;
      x[3] = b;
    }
  }
}

// kTA / kTB: A stored K x M / B stored N x K, staged by the transposing
// cp.async copies.  kTma: the operands that are not transposed come by TMA
// (all others by cp.async); with one operand transposed the two kinds of
// copy complete on the same mbarrier (1 TMA arrival + 256 cp.async ones).
// kCT: C is stored transposed (p.c_trans), a compile-time choice so that the
// row-major instances carry no trace of it.  kPairK: the grid of two CTAs
// per tile over the two halves of K (SgemmParams::cluster_k), launched as
// clusters of two.
template <bool kTma, int TN, int kMinBlocks, bool kTA = false, bool kTB = false, bool kCT = false,
          bool kPairK = false>
__global__ void __launch_bounds__(kSgemmThreads, kMinBlocks)
    sgemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const SgemmParams p) {
  static_assert(!(kTma && kTA && kTB), "with both operands transposed nothing is TMA-staged");
  static_assert(!(kPairK && (kTA || kTB || kCT)), "CTA pairs over K take row-major operands");
  constexpr bool kCpA = !kTma || kTA;   // A staged by cp.async
  constexpr bool kCpB = !kTma || kTB;   // B staged by cp.async
  constexpr bool kAnyCp = kCpA || kCpB;
  constexpr uint32_t kBarCount = (kTma ? 1u : 0u) + (kAnyCp ? (uint32_t)kSgemmThreads : 0u);
  constexpr int BN = sgemm_bn(TN);
  constexpr int S = sgemm_stages(sgemm_cfg(TN, kMinBlocks));
  constexpr int kRelease = S - 1;   // k-tiles per ring release (see the k-loop)
  static_assert(kRelease >= 2, "the ring has at least three stages");
  constexpr int kBStageFloats = BK * BN;
  constexpr int NH = TN / 4;   // 16-byte column groups per thread

  extern __shared__ unsigned char smem_raw[];
  __shared__ int s_abort;
  __shared__ int s_second;   // this CTA's cut piece got to its tile second
  unsigned char* const base = align_smem_1024(smem_raw);
  float* sA = reinterpret_cast<float*>(base);
  float* sB = sA + S * kAStageFloats;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + S * kBStageFloats);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), kBarCount);
    s_abort = 0;
    fence_mbar_init();
    if constexpr (!kCpA) tma_prefetch_desc(&tmA);
    if constexpr (!kCpB) tma_prefetch_desc(&tmB);
  }
  __syncthreads();
  wait_prior_grids();
  allow_dependent_grids();

  // Thread -> output mapping.  Warp (warp_m, warp_n) owns a 32 x (BN/2)
  // block; lane (tr, tc) owns rows tr + 4i (i < 8) and columns
  // tc*4 + 32h + {0..3} (h < TN/4) of it.
  // Each group of 4 consecutive lanes is a 2 x 2 block of (tr, tc): a
  // shared-memory wavefront delivers one distinct 16-byte chunk to each
  // 4-lane group, so a 16-byte fragment load costs the minimum 2 wavefronts
  // only if the group touches at most 2 chunks (2 A rows, 2 B column groups).
  const int warp_m = warp >> 1;
  const int warp_n = warp & 1;
  const int tr = ((lane >> 4) << 1) | ((lane >> 1) & 1);       // 0..3
  const int tc = (((lane >> 2) & 3) << 1) | (lane & 1);        // 0..7
  const int a_row0 = warp_m * 32 + tr;            // row for i = 0
  const int b_col0 = warp_n * (BN / 2) + tc * 4;

  // Work of this CTA.  Split-K mode (slices > 1): one unit, k-slice
  // b % slices of tile b / slices.  Otherwise (hybrid stream-K, G =
  // gridDim.x): first whole tiles b, b + G, ... below dp_tiles (full waves in
  // tile order, so the tiles in flight together are neighbours and share
  // A and B in L2), then the k-tiles [b * total / G, (b + 1) * total / G) of
  // the remaining tiles' (tile, k-tile) iteration space, total =
  // (tiles - dp_tiles) * nk_all, as one unit per tile they touch.  The host
  // keeps G <= tiles - dp_tiles, so each range covers at least one tile's
  // worth of k-tiles, or G = 2 tiles, so each range is half a tile: either
  // way a tile is cut into at most two pieces.  The ring's slot and phase
  // follow the k-tiles this CTA has consumed over all its units (g0 + kt).
  //
  // Within its range a CTA runs its whole tiles first, then the head of the
  // last tile it touches (k-tiles from 0), then the tail of the first (up to
  // nk): every CTA then works at k-tile tau or tau - (share mod nk) of its
  // units at time tau, so the share's A and B panels are read in two fronts
  // instead of at as many k offsets as there are CTAs, and L2 holds the
  // slices in between (the two pieces of a cut tile combine in whichever
  // order they finish, see below).  Measured on GB300 at 4096^3: DRAM
  // traffic 435 -> 389 MB per launch, same time.
  const int nk_all = (p.K + BK - 1) / BK;
  const int b = blockIdx.x;
  int dp_next = b;
  int sk_units = 0, sk_next = 0;   // stream-K units of this CTA, the next one
  int sk_t0 = 0, sk_kb0 = 0, sk_t1 = 0, sk_ke1 = 0, sk_w0 = 0, sk_nw = 0;
  bool sk_head = false;
  if (p.slices > 1) {
    dp_next = 0x7fffffff;
    sk_units = 1;
  } else {
    const long long total = (long long)(p.tiles_m * p.tiles_n - p.dp_tiles) * nk_all;
    const long long it0 = (long long)b * total / gridDim.x;
    const long long it1 = (long long)(b + 1) * total / gridDim.x;
    if (it1 > it0) {
      sk_t0 = (int)(it0 / nk_all);
      sk_kb0 = (int)(it0 % nk_all);
      sk_t1 = (int)((it1 - 1) / nk_all);
      sk_ke1 = (int)((it1 - 1) % nk_all) + 1;
      if (sk_t0 == sk_t1) {
        sk_units = 1;   // half a tile: one unit [kb0, ke1)
      } else {
        sk_head = sk_ke1 < nk_all;
        sk_w0 = sk_t0 + (sk_kb0 > 0 ? 1 : 0);
        sk_nw = sk_t1 - (sk_head ? 1 : 0) - sk_w0 + 1;
        sk_units = sk_nw + (sk_head ? 1 : 0) + (sk_kb0 > 0 ? 1 : 0);
      }
    }
  }
  int g0 = 0;
  bool pair_synced = false;   // kPairK: this CTA passed the exchange's two cluster barriers
  while (dp_next < p.dp_tiles || sk_next < sk_units) {
    int tile, k_begin, k_end;
    if (p.slices > 1) {
      tile = b / p.slices;
      const int sl = b - tile * p.slices;
      k_begin = sl * nk_all / p.slices;
      k_end = (sl + 1) * nk_all / p.slices;
      ++sk_next;
    } else if (dp_next < p.dp_tiles) {
      tile = dp_next;
      k_begin = 0;
      k_end = nk_all;
      dp_next += gridDim.x;
    } else {
      const int u = sk_next++;
      int t;
      if (sk_t0 == sk_t1) {
        t = sk_t0;
        k_begin = sk_kb0;
        k_end = sk_ke1;
      } else if (u < sk_nw) {
        t = sk_w0 + u;
        k_begin = 0;
        k_end = nk_all;
      } else if (sk_head && u == sk_nw) {
        t = sk_t1;
        k_begin = 0;
        k_end = sk_ke1;
      } else {
        t = sk_t0;
        k_begin = sk_kb0;
        k_end = nk_all;
      }
      tile = p.dp_tiles + t;
    }
    int tm, tn;
    grouped_tile(tile, p.tiles_m, p.tiles_n, kSgemmGroupM, tm, tn);
    const int m0 = tm * BM;
    const int n0 = tn * BN;
    const int nk = k_end - k_begin;   // k-tiles of this unit

    // Stage k-tile kt (counted from k_begin) into ring slot s.
    auto issue = [&](int kt, int s) {
      const int k0 = (k_begin + kt) * BK;
      const uint32_t bar = smem_u32(&full[s]);
      if constexpr (kTma) {
        if (tid == 0) {
          mbar_arrive_expect_tx(bar, (kCpA ? 0u : kAStageFloats * 4u) +
                                         (kCpB ? 0u : (uint32_t)kBStageFloats * 4u));
          if constexpr (!kCpA) tma_load_operand<0>(smem_u32(sA + s * kAStageFloats), &tmA, bar, k0, m0);
          if constexpr (!kCpB) tma_load_operand<1>(smem_u32(sB + s * kBStageFloats), &tmB, bar, n0, k0);
        }
      }
      if constexpr (kAnyCp) {
        const uint32_t a_dst = smem_u32(sA + s * kAStageFloats);
        if constexpr (!kCpA) {
          // A comes by TMA.
        } else if constexpr (!kTA) {
          // A: a warp copies one 32-float row segment (k contiguous in memory).
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
        } else {
          // A stored K x M (m contiguous): copy j of warp w covers m = 8 g + (lane
          // mod 8), k = 4 q + lane / 8 with g = (16 w + j) / 8, q = (16 w + j) mod 8.
  #pragma unroll
          for (int j = 0; j < BM * BK / (32 * 8); ++j) {
            const int idx = (BM * BK / (32 * 8)) * warp + j;
            const int m = 8 * (idx >> 3) + (lane & 7);
            const int k = 4 * (idx & 7) + (lane >> 3);
            const int gm = m0 + m;
            const int gk = k0 + k;
            const bool v = (gm < p.M) && (gk < p.K);
            const float* src = v ? p.A + (long long)gk * p.lda + gm : p.A;
            cp_async_4(a_dst + 4u * a_tile_offset(m, k), src, v);
          }
        }
        const uint32_t b_dst = smem_u32(sB + s * kBStageFloats);
        if constexpr (!kCpB) {
          // B comes by TMA.
        } else if constexpr (!kTB) {
          // B: BN consecutive threads copy one BN-float row segment.
          constexpr int kRowsPerPass = kSgemmThreads / BN;
          const int nb = tid % BN;
          const int gn = n0 + nb;
  #pragma unroll
          for (int j = 0; j < BK / kRowsPerPass; ++j) {
            const int k = tid / BN + kRowsPerPass * j;
            const int gk2 = k0 + k;
            const bool v = (gk2 < p.K) && (gn < p.N);
            const float* src = v ? p.B + (long long)gk2 * p.ldb + gn : p.B;
            cp_async_4(b_dst + 4u * b_tile_offset(BN, k, nb), src, v);
          }
        } else {
          // B stored N x K (k contiguous): copy j of warp w covers n = 4 g +
          // lane / 8, k = 4 (lane mod 8) + kk with g = (BN/32) w + j / 4 and
          // kk = j mod 4; the four copies of one g read the same four rows.
          constexpr int kPer = BN * BK / (32 * 8);   // copies per thread
  #pragma unroll
          for (int j = 0; j < kPer; ++j) {
            const int n = 4 * ((BN / 32) * warp + (j >> 2)) + (lane >> 3);
            const int k = 4 * (lane & 7) + (j & 3);
            const int gn = n0 + n;
            const int gk = k0 + k;
            const bool v = (gn < p.N) && (gk < p.K);
            const float* src = v ? p.B + (long long)gn * p.ldb + gk : p.B;
            cp_async_4(b_dst + 4u * bt_tile_offset(BN, k, n), src, v);
          }
        }
        cp_async_mbar_arrive_noinc(bar);
      }
    };

    const int pre = nk < S ? nk : S;
    for (int kt = 0; kt < pre; ++kt) issue(kt, (g0 + kt) % S);

    // acc[i][j] holds columns (2j, 2j+1) of row i as a packed float pair.
    unsigned long long acc[8][TN / 2];
  #pragma unroll
    for (int i = 0; i < 8; ++i)
  #pragma unroll
      for (int j = 0; j < TN / 2; ++j) acc[i][j] = 0ull;

    int kt = 0;
    for (; kt < nk; ++kt) {
      const int s = (g0 + kt) % S;
      const bool ok = mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)(((g0 + kt) / S) & 1),
                                        p.timeout_ns, &s_abort);
      if (!ok) {
        s_abort = 1;
      } else {
        const float* As = sA + s * kAStageFloats + a_row0 * BK;
        // (A transposed-B tile has the thread's column chunk tc XOR-ed with kq.)
        const float* Bs = sB + s * kBStageFloats + (kTB ? b_col0 - 4 * tc : b_col0);
        // Row (a_row0 + 4i) mod 8 = tr + 4 (i mod 2), so k-quad kq of the
        // thread's even rows sits in chunk kq ^ tr, of its odd rows in chunk
        // kq ^ tr ^ 4.  Four base pointers cover (kq mod 4) ^ tr.
        const float* a_base[4];
  #pragma unroll
        for (int q = 0; q < 4; ++q) a_base[q] = As + (((q ^ tr) & 3) << 2);
  #pragma unroll
        for (int kq = 0; kq < BK / 4; ++kq) {
          // A fragment: four k-steps of each of the thread's 8 rows.
          float4 a[8];
  #pragma unroll
          for (int i = 0; i < 8; ++i)
            a[i] = *reinterpret_cast<const float4*>(a_base[kq & 3] + 4 * i * BK +
                                                    (((kq & 4) ^ ((i & 1) << 2)) << 2));
  #pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const float* brow = Bs + (kq * 4 + kk) * BN + (kTB ? ((tc ^ kq) << 2) : 0);
            ulonglong2 b[NH];
  #pragma unroll
            for (int h = 0; h < NH; ++h) b[h] = lds128_pairs(brow + 32 * h);
            // All eight broadcast A pairs first, then the FFMA2s with the B
            // column group outermost: the first group needs only b[0], so
            // the FMA pipe starts before the other fragment loads land
            // (measured 2184 -> 2100 us at 4096^3 against row-outermost).
            unsigned long long aa[8];
  #pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float av = (&a[i].x)[kk];
              aa[i] = pack_pair(av, av);
            }
  #pragma unroll
            for (int h = 0; h < NH; ++h) {
  #pragma unroll
              for (int i = 0; i < 8; ++i) {
                ffma2(acc[i][2 * h + 0], aa[i], b[h].x);
                ffma2(acc[i][2 * h + 1], aa[i], b[h].y);
              }
            }
          }
        }
      }
      // Slots are released kRelease = S - 1 k-tiles at a time (one
      // barrier per kRelease k-tiles, at least one k-tile always in flight):
      // at the end of each group every thread is done with the group's
      // slots, whose k-tiles + S are staged now; the last k-tile ends with
      // a barrier too (or some thread gave up).
      const bool group_end = (kt + 1) % kRelease == 0;
      if (group_end || kt + 1 == nk) {
        if (__syncthreads_or(!ok || *(volatile int*)&s_abort)) break;
        if (group_end) {
  #pragma unroll
          for (int r = kRelease - 1; r >= 0; --r)
            if (kt - r + S < nk) issue(kt - r + S, (g0 + kt - r) % S);
        }
      }
    }

    if (kt < nk) {
      // A wait gave up: record it, let this CTA's own copies land, and leave
      // without writing C.
      if (tid == 0) raise_fault(p.fault, kFaultSgemmFullWait);
      if constexpr (kAnyCp) cp_async_wait_all();
      if constexpr (kTma) {
        if (tid == 0) {
          // The last release point followed k-tile `from` - 1 (the start
          // of kt's group) and staged up to that + S; every k-tile from
          // `from` on may still be in flight.
          const int from = kt / kRelease * kRelease;
          const int issued = from + S < nk ? from + S : nk;
          for (int t = from; t < issued; ++t) {
            if (!mbar_wait_bounded(smem_u32(&full[(g0 + t) % S]), (uint32_t)(((g0 + t) / S) & 1),
                                   p.timeout_ns, nullptr)) {
              raise_fault(p.fault, kFaultDrainWait);
              break;
            }
          }
        }
      }
      __syncthreads();
      // (The partner CTA of a pair waits at two cluster barriers: pass them.)
      if constexpr (kPairK) {
        cluster_sync_all();
        cluster_sync_all();
      }
      return;
    }

    if constexpr (kPairK) {
      // The two CTAs of this tile's cluster hold the sums over the two
      // halves of K (rank 0 the first).  Rank 0 keeps rows 0..63 (warps
      // 0..3) and rank 1 rows 64..127 (warps 4..7); each warp of the other
      // half sends its accumulators into the partner's (now idle) ring,
      // where the warp with the same rows adds them to its own and the
      // tile's C is written half by each CTA.  Thread t (mod 128) puts its
      // j-th 16-byte group at ring + 16 (128 j + t): a warp's stores and
      // loads are contiguous, free of bank conflicts.  a + b == b + a, so
      // the result does not depend on which half is whose.
      const uint32_t rank = (uint32_t)b & 1u;
      const bool keep = (warp_m < 2) == (rank == 0);
      const int t = tid & 127;
      cluster_sync_all();   // both CTAs are done with their rings
      if (!keep) {
        const uint32_t dst = mapa_shared(smem_u32(sA), rank ^ 1u);
  #pragma unroll
        for (int i = 0; i < 8; ++i) {
  #pragma unroll
          for (int h = 0; h < NH; ++h) {
            const float2 lo = unpack_pair(acc[i][2 * h + 0]);
            const float2 hi = unpack_pair(acc[i][2 * h + 1]);
            st_cluster_v4(dst + 16u * (uint32_t)(128 * (i * NH + h) + t), lo.x, lo.y, hi.x, hi.y);
          }
        }
      }
      cluster_sync_all();   // the partner's half is in this CTA's ring
      pair_synced = true;
      if (!keep) {
        g0 += nk;
        continue;
      }
  #pragma unroll
      for (int i = 0; i < 8; ++i) {
  #pragma unroll
        for (int h = 0; h < NH; ++h) {
          const float4 o = *reinterpret_cast<const float4*>(sA + 4 * (128 * (i * NH + h) + t));
          const float2 lo = unpack_pair(acc[i][2 * h + 0]);
          const float2 hi = unpack_pair(acc[i][2 * h + 1]);
          acc[i][2 * h + 0] = pack_pair(lo.x + o.x, lo.y + o.y);
          acc[i][2 * h + 1] = pack_pair(hi.x + o.z, hi.y + o.w);
        }
      }
    }

    // Destination: unscaled FP32 partial sums go to
    // part[(gm - part_m0) * part_ld + gn - part_n0]; add_into_c pieces add
    // into C; everything else is stored to C.
    float* part = nullptr;
    long long part_ld = 0;
    int part_m0 = 0, part_n0 = 0;
    bool add_into_c = false;
    unsigned* done_flag = nullptr;   // set to p.epoch once this unit's stores are visible
    if (p.slices > 1) {
      part = p.ws + (long long)(b % p.slices) * p.M * p.ldw;
      part_ld = p.ldw;
    } else if (!kPairK && (k_begin != 0 || k_end != nk_all)) {
      // One of the two pieces of a tile cut by boundary cb (the first k-tile
      // of CTA cb): piece 0 ends CTA cb - 1's range, piece 1 starts CTA cb's.
      // Whichever piece finishes first publishes its sums and raises the
      // boundary's done flag; the second waits for that flag (the first has
      // already finished its k-loop, so the wait is short and needs no
      // co-residency) and completes the tile.  With beta == 0 the first
      // stores alpha * sums to C and the second adds alpha * its sums into
      // it; otherwise the first leaves its unscaled sums in the boundary's
      // workspace tile and the second adds them to its accumulators and
      // writes alpha * total + beta * C.  Two addends give the same sum in
      // either order, so the result does not depend on which came first.
      const int cb = k_begin == 0 ? b + 1 : b;
      unsigned* arrive = p.sk_flags + 2 * (cb - 1);
      if (tid == 0) {
        const bool second = atomicExch(arrive, p.epoch) == p.epoch;
        if (second) {
          if (!flag_wait_equal(arrive + 1, p.epoch, p.timeout_ns, nullptr))
            raise_fault(p.fault, kFaultSgemmPieceWait);
          // The first piece is done with both words: clear them, so that a
          // replay of this launch (a CUDA graph, same epoch) starts afresh.
          arrive[0] = 0u;
          arrive[1] = 0u;
        }
        s_second = second ? 1 : 0;
      }
      __syncthreads();
      float* const slot =
          p.tail_ws != nullptr ? p.tail_ws + (long long)(cb - 1) * (BM * BN) : nullptr;
      if (!s_second) {
        done_flag = arrive + 1;
        if (slot != nullptr) {
          part = slot;
          part_ld = BN;
          part_m0 = m0;
          part_n0 = n0;
        }
      } else if (slot != nullptr) {
        // (The slot holds the first piece's sums at every element of the
        // tile inside C; the others are never stored.)
  #pragma unroll
        for (int i = 0; i < 8; ++i) {
  #pragma unroll
          for (int h = 0; h < NH; ++h) {
            const float4 o = __ldcg(reinterpret_cast<const float4*>(
                slot + (a_row0 + 4 * i) * BN + b_col0 + 32 * h));
            const float2 lo = unpack_pair(acc[i][2 * h + 0]);
            const float2 hi = unpack_pair(acc[i][2 * h + 1]);
            acc[i][2 * h + 0] = pack_pair(lo.x + o.x, lo.y + o.y);
            acc[i][2 * h + 1] = pack_pair(hi.x + o.z, hi.y + o.w);
          }
        }
      } else {
        add_into_c = true;
      }
    }
    // After the first piece's stores: make them visible, then raise the flag.
    const auto publish = [&]() {
      if (done_flag == nullptr) return;
      __threadfence();
      __syncthreads();
      if (tid == 0) flag_store_release(done_flag, p.epoch);
    };

    // Scaling pass, C := alpha * (A.B) + beta * C, applied to the
    // accumulators in place before any store (partial sums for a workspace
    // stay unscaled).  The old C of one row (TN values) is loaded at once so
    // that those loads overlap instead of each waiting behind a store.
    if (!kCT && part == nullptr && (p.alpha != 1.f || p.beta != 0.f)) {
      const bool vec4c = p.c_vec4 != 0;
  #pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int gm = m0 + a_row0 + 4 * i;
        const float* crow = p.C + (long long)gm * p.ldc;
        float4 old[NH];
  #pragma unroll
        for (int h = 0; h < NH; ++h) {
          const int gn = n0 + b_col0 + 32 * h;
          float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
          if (p.beta != 0.f && gm < p.M) {
            if (vec4c && gn + 3 < p.N) {
              c = *reinterpret_cast<const float4*>(crow + gn);
            } else {
              if (gn + 0 < p.N) c.x = crow[gn + 0];
              if (gn + 1 < p.N) c.y = crow[gn + 1];
              if (gn + 2 < p.N) c.z = crow[gn + 2];
              if (gn + 3 < p.N) c.w = crow[gn + 3];
            }
          }
          old[h] = c;
        }
  #pragma unroll
        for (int h = 0; h < NH; ++h) {
          const float2 lo = unpack_pair(acc[i][2 * h + 0]);
          const float2 hi = unpack_pair(acc[i][2 * h + 1]);
          // (A column past N got c = 0 and is never stored.)
          const auto upd = [&](float v, float cv) {
            return p.beta != 0.f ? fmaf(p.beta, cv, p.alpha * v) : p.alpha * v;
          };
          acc[i][2 * h + 0] = pack_pair(upd(lo.x, old[h].x), upd(lo.y, old[h].y));
          acc[i][2 * h + 1] = pack_pair(upd(hi.x, old[h].z), upd(hi.y, old[h].w));
        }
      }
    }

    if (kCT && part == nullptr) {
      // C stored transposed: the kernel's element (gm, gn) is
      // C[gn * ldc + gm], so a column of the tile is a row of C.  For each
      // of its columns a thread holds rows tr + 4i; transposing among the
      // four lanes of equal tc gives each lane four consecutive rows, stored
      // (or, for a stream-K piece, added) as one 16-byte access, so a warp
      // store writes whole 32-byte sectors.  C := alpha * (A.B) + beta * C
      // is applied here, on the same 16 bytes.
      const bool v4 = p.c_vec4 != 0;
      const int gm_blk = m0 + a_row0 - tr;
  #pragma unroll
      for (int h = 0; h < NH; ++h) {
  #pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int gn = n0 + b_col0 + 32 * h + q;
  #pragma unroll
          for (int u = 0; u < 2; ++u) {
            float x[4];
  #pragma unroll
            for (int s = 0; s < 4; ++s) {
              const float2 pr = unpack_pair(acc[4 * u + s][2 * h + (q >> 1)]);
              x[s] = (q & 1) ? pr.y : pr.x;
            }
            transpose4_lanes(x, tr);
            const int gm = gm_blk + 16 * u + 4 * tr;
            if (gn >= p.N) continue;
            float* dst = p.C + (long long)gn * p.ldc + gm;
            if (v4 && gm + 3 < p.M) {
              float4 v = make_float4(p.alpha * x[0], p.alpha * x[1], p.alpha * x[2],
                                     p.alpha * x[3]);
              if (add_into_c) {
                atomicAdd(reinterpret_cast<float4*>(dst), v);
              } else {
                if (p.beta != 0.f) {
                  const float4 o = *reinterpret_cast<const float4*>(dst);
                  v = make_float4(fmaf(p.beta, o.x, v.x), fmaf(p.beta, o.y, v.y),
                                  fmaf(p.beta, o.z, v.z), fmaf(p.beta, o.w, v.w));
                }
                *reinterpret_cast<float4*>(dst) = v;
              }
            } else {
  #pragma unroll
              for (int r = 0; r < 4; ++r) {
                if (gm + r >= p.M) break;
                float v = p.alpha * x[r];
                if (add_into_c) {
                  atomicAdd(dst + r, v);
                } else {
                  if (p.beta != 0.f) v = fmaf(p.beta, dst[r], v);
                  dst[r] = v;
                }
              }
            }
          }
        }
      }
      publish();
      g0 += nk;
      continue;
    }

    // Epilogue: each store instruction of a warp covers four full 128-byte row
    // segments of C.
  #pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int gm = m0 + a_row0 + 4 * i;
      if (gm >= p.M) continue;
      // Column gn of this row is crow[gn - cshift] (element by element at
      // c_index for a transposed C).
      float* crow = part != nullptr ? part + (long long)(gm - part_m0) * part_ld
                                    : p.C + (long long)gm * p.ldc;
      const int cshift = part_n0;
      const bool vec4 = part != nullptr ? true : (p.c_vec4 != 0 && !kCT);
      const auto elem = [&](int col) {
        if constexpr (kCT)
          return part != nullptr ? crow + col - cshift : p.C + kc_index<kCT>(p, gm, col);
        else
          return crow + col - cshift;
      };
  #pragma unroll
      for (int h = 0; h < NH; ++h) {
        const int gn = n0 + b_col0 + 32 * h;
        const float2 lo = unpack_pair(acc[i][2 * h + 0]);
        const float2 hi = unpack_pair(acc[i][2 * h + 1]);
        const float v0 = lo.x, v1 = lo.y, v2 = hi.x, v3 = hi.y;
        if (add_into_c) {
          if (vec4 && gn + 3 < p.N) {
            atomicAdd(reinterpret_cast<float4*>(crow + gn), make_float4(v0, v1, v2, v3));
          } else {
            if (gn + 0 < p.N) atomicAdd(elem(gn + 0), v0);
            if (gn + 1 < p.N) atomicAdd(elem(gn + 1), v1);
            if (gn + 2 < p.N) atomicAdd(elem(gn + 2), v2);
            if (gn + 3 < p.N) atomicAdd(elem(gn + 3), v3);
          }
        } else if (vec4 && gn + 3 < p.N) {
          *reinterpret_cast<float4*>(crow + gn - cshift) = make_float4(v0, v1, v2, v3);
        } else {
          if (gn + 0 < p.N) *elem(gn + 0) = v0;
          if (gn + 1 < p.N) *elem(gn + 1) = v1;
          if (gn + 2 < p.N) *elem(gn + 2) = v2;
          if (gn + 3 < p.N) *elem(gn + 3) = v3;
        }
      }
    }
    publish();
    g0 += nk;
  }
  // A CTA of a pair with no unit (never planned) still meets its partner's
  // two cluster barriers.
  if constexpr (kPairK) {
    if (!pair_synced) {
      cluster_sync_all();
      cluster_sync_all();
    }
  }
}

template <bool kTma, int TN, int kMinBlocks, bool kTA = false, bool kTB = false, bool kCT = false,
          bool kPairK = false>
cudaError_t launch_cfg(const SgemmParams& p, const CUtensorMap* tmA, const CUtensorMap* tmB,
                       cudaStream_t stream) {
  // The attribute is per function; setting it on every call is cheap and
  // keeps this correct for every device of the process.
  const auto kernel = sgemm_kernel<kTma, TN, kMinBlocks, kTA, kTB, kCT, kPairK>;
  constexpr int kSmem = sgemm_smem_bytes(sgemm_cfg(TN, kMinBlocks));
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const int tiles = p.tiles_m * p.tiles_n;
  // Stream-K: G = p.grid CTAs (<= tiles); p.split_tiles tiles are cut in two.
  const int G = p.slices > 1 ? tiles * p.slices : p.grid;
  return launch_gemm_kernel_clusters(kPairK ? 2u : 1u, kernel, dim3(G), dim3(kSgemmThreads),
                                     kSmem, stream, *tmA, *tmB, p);
}

}  // namespace

}  // namespace dgemm
