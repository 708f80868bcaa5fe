// FP16 / BF16 GEMM on sm_103a tensor cores with CTA pairs: C = A . B,
// row-major, FP32 accumulation in tensor memory, FP16 / BF16 output rounded to
// nearest-even.
//
// Same five-step flow as the single-CTA kernel (GB300 GEMM roadmap,
// m.nxbn.cn, section 4.2: TMA -> shared memory -> tcgen05.mma into TMEM ->
// tcgen05.ld -> epilogue), and the same reading of its section 1.1 that the
// data supply limits a GEMM here: a trace of the single-CTA kernel showed
// its MMA thread waiting for loaded stages 27-29 % of the time, with a
// 4-stage ring of 48 KB stages being all the shared memory there is.
//
// A cluster of two CTAs on two SMs computes a 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256): each CTA stages its own 128 rows of A
// and its own half (128 columns) of B, and the MMA reads the peer's half
// through the cluster.  Per SM and 64 of K that is 32 KB instead of 48 KB,
// so each SM fetches a third fewer operand bytes per FLOP.  A ring stage is
// 128 deep (64 KB, three stages): one barrier wait, fence and commit covers
// eight MMAs (a %globaltimer trace had put ~43 % of the MMA issuer's loop in
// that per-stage bookkeeping with 64-deep stages).
//
// Roles per CTA (192 threads): warp 0 TMA producer, warp 1 TMEM allocator
// (both CTAs) and MMA issuer (even CTA only, one thread), warps 2-5 epilogue
// (each CTA drains its own 128 TMEM lanes).  Barriers:
//  * full[s]   (even CTA): both CTAs' TMA loads complete on it; the even
//              CTA's producer posts the pair's byte count;
//  * empty[s]  (each CTA): arrived by a multicast tcgen05.commit once the
//              MMAs reading stage s are done;
//  * acc_full  (each CTA): multicast commit after a unit's last k-tile;
//  * acc_empty (even CTA): both CTAs' epilogue warps arrive (8 arrivals).
// The tiles of a last partial round run as two 128-column parts.  Every
// wait is bounded; a wait that gives up records a fault and the roles unwind.
// Operands stored transposed (kAT, kBT) are read as stored, as in the
// single-CTA kernel: an MN-major A (two 64-row blocks per CTA) and a K-major
// B (the CTA's 128 columns as 128 rows of 64 k).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "launch.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace dgemm {
namespace {

constexpr int BM = kTc2BM;            // rows per CTA (256 per pair)
constexpr int BN = kTc2BN;            // columns per pair tile
constexpr int BK = kTc2BK;
constexpr int S = kTc2Stages;
constexpr int UMMA_K = 16;
constexpr uint32_t kABytes = BM * BK * 2;          // 32 KB
constexpr uint32_t kBBoxBytes = 64 * BK * 2;       // one 64-column block of B: 16 KB
constexpr uint32_t kBBytes = (BN / 2) * BK * 2;    // this CTA's half of B: 32 KB
// A stage holds BK / 64 k-blocks of 64: a K-major operand keeps each as its
// own 128-byte-swizzled tile (rows x 128 bytes), kAKBlock / kBKBlock bytes
// apart; an MN-major operand keeps BK rows of 128 bytes per 64-wide block,
// kMNBlock bytes apart.  Every TMA box is 64 k deep (the tensor maps are the
// single-CTA kernel's), so a stage takes BK / 64 boxes per block.
constexpr int kKBlocks = BK / 64;
constexpr uint32_t kAKBlock = BM * 128;            // 16 KB
constexpr uint32_t kBKBlock = (BN / 2) * 128;      // 16 KB
constexpr uint32_t kMNBlock = BK * 128;            // 16 KB
constexpr uint32_t kBox64 = 64 * 128;              // one 64 x 64 box: 8 KB
constexpr uint32_t kEpiBufBytes = 32 * kTcEpiCols * 2;
constexpr int kAccBufs = kTc2AccBufs;              // accumulator buffers in TMEM
constexpr uint32_t kTmemCols = kAccBufs * BN;
constexpr int kEpiWarps = 4;

static_assert(BK % 64 == 0, "a stage is whole 64-deep swizzle blocks");
static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM allocations are powers of two");

struct alignas(8) Barriers {
  uint64_t full[S];
  uint64_t empty[S];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// The FP32 head partial of boundary `slot`, CTA `rank`, epilogue warp q:
// 32 rows x 256 columns, lane-major: the 16-byte group g (columns 4g ..
// 4g + 3) of lane l's row lands at (g * 32 + l) x 4 floats from the block
// start, so that a warp's store or load of one g is 512 contiguous bytes.
__device__ __forceinline__ float* partial_block(const TcParams& p, int slot, int rank, int q) {
  const long long blk = ((long long)slot * 2 + rank) * 4 + q;
  return p.kpart + blk * (32 * BN);
}
__device__ __forceinline__ unsigned* partial_flag(const TcParams& p, int slot, int rank, int q) {
  return p.kflag + (((long long)slot * 2 + rank) * 4 + q);
}

// A single thread's bounded wait (the MMA issuer's): spins on the barrier;
// on giving up records the fault (once per CTA) and raises the abort flag.
__device__ __forceinline__ bool thread_wait(uint32_t bar, uint32_t parity, const TcParams& p,
                                            Barriers* bars, unsigned fault_code) {
  if (mbar_wait_spin_bounded(bar, parity, p.timeout_ns, &bars->abort)) return true;
  if (!*(volatile int*)&bars->abort) raise_fault(p.fault, fault_code);
  *(volatile int*)&bars->abort = 1;
  return false;
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const TcParams& p,
                                          Barriers* bars, unsigned fault_code) {
  const int lane = threadIdx.x & 31;
  int ok = 1;
  if (lane == 0) {
    // The producer and the MMA issuer spin; the epilogue warps, which wait a
    // whole tile for an accumulator, suspend.
    const bool got = fault_code == kFaultTcEpilogueWait
                         ? mbar_wait_bounded(bar, parity, p.timeout_ns, &bars->abort)
                         : mbar_wait_spin_bounded(bar, parity, p.timeout_ns, &bars->abort);
    ok = got ? 1 : 0;
    if (!ok) {
      if (!*(volatile int*)&bars->abort) raise_fault(p.fault, fault_code);
      *(volatile int*)&bars->abort = 1;
    }
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <typename T, uint32_t kAbType, bool kAT, bool kBT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kTcThreads, 1)
    gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* const base = align_smem_1024(smem_raw);
  unsigned char* sA = base;
  unsigned char* sB = sA + S * kABytes;
  unsigned char* sEpi = sB + S * kBBytes;
  Barriers* bars = reinterpret_cast<Barriers*>(sEpi + kEpiWarps * 2 * kEpiBufBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();     // 0: issues the MMAs
  const int npairs = gridDim.x >> 1;
  const int nk = (p.K + BK - 1) / BK;
  const TcPairSched sched = tc_pair_sched(blockIdx.x >> 1, npairs, p, nk);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars->acc_full[b]), 1);
      mbar_init(smem_u32(&bars->acc_empty[b]), 2 * kEpiWarps);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(&bars->tmem_base), kTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();     // the peer's barriers are initialised
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;
  wait_prior_grids();
  allow_dependent_grids();
  if (rank == 1 && threadIdx.x == 0) {
    // The pair's MMAs address both CTAs' TMEM at the even CTA's base.
    uint32_t leader_base;
    asm volatile("ld.shared::cluster.u32 %0, [%1];"
                 : "=r"(leader_base)
                 : "r"(mapa_shared(smem_u32(&bars->tmem_base), 0)));
    if (leader_base != tmem_base) raise_fault(p.fault, kFaultTcPairTmem);
  }

  uint32_t issued = 0;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    uint32_t it = 0;
    bool ok = true;
    for (int j = 0; j < sched.n && ok; ++j) {
      const TcUnit w = tc_pair_unit(sched, j, npairs, p, nk);
      const int half = w.n_w / 2;          // columns of B this CTA stages
      const int boxes = half / 64;
      for (int kt = w.kb; kt < w.ke; ++kt, ++it) {
        const uint32_t s = it % S;
        const uint32_t ph = (it / S) & 1u;
        ok = warp_wait(smem_u32(&bars->empty[s]), ph ^ 1u, p, bars, kFaultTcProducerWait);
        if (!ok) break;
        if (lane == 0) {
          const uint32_t fb = mapa_shared(smem_u32(&bars->full[s]), 0);
          if (rank == 0)
            mbar_arrive_expect_tx(smem_u32(&bars->full[s]), 2 * (kABytes + boxes * kBBoxBytes));
          const uint32_t adst = smem_u32(sA + s * kABytes);
          const uint32_t bdst = smem_u32(sB + s * kBBytes);
          const int m = w.tm * (2 * BM) + (int)rank * BM;
          for (int kb = 0; kb < kKBlocks; ++kb) {
            const int k = kt * BK + kb * 64;
            if constexpr (!kAT) {   // K-major: one 128-row box per k-block
              tma_load_operand_pair<0>(adst + kb * kAKBlock, &tmA, fb, k, m);
            } else {   // A stored K x M: two 64-row (m) blocks, MN-major
              for (int jj = 0; jj < BM / 64; ++jj)
                tma_load_operand_pair<0>(adst + jj * kMNBlock + kb * kBox64, &tmA, fb, m + jj * 64, k);
            }
            if constexpr (kBT) {   // B stored N x K: 64 rows (n) of 64 k per box, K-major
              for (int jj = 0; jj < boxes; ++jj) {
                const int n = w.tn * BN + w.n_off + (int)rank * half + jj * 64;
                tma_load_operand_pair<1>(bdst + kb * kBKBlock + jj * kBox64, &tmB, fb, k, n);
              }
            }
          }
          if constexpr (!kBT) {   // MN-major: one box per 64-column block, all BK rows
            for (int jj = 0; jj < boxes; ++jj) {
              const int n = w.tn * BN + w.n_off + (int)rank * half + jj * 64;
              tma_load_operand_pair<1>(bdst + jj * kMNBlock, &tmB, fb, n, kt * BK);
            }
          }
          issued = it + 1;
        }
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (even CTA)
    // One thread issues every MMA of the pair and waits on the barriers by
    // itself.  A tcgen05.mma is accepted about as fast as the tensor pipe
    // runs it, so the thread is busy for most of a stage; any warp-wide
    // synchronisation between stages (a shuffle of the wait's result, a
    // __syncwarp) left the pipe idle for ~0.2 us per stage -- 22 % of the
    // MMA time, measured with the operand loads removed.
    // (Waiting for the next stage before committing the current one, to
    // keep the wait off the pipe's path, was measured slower: 92.9 vs 88.7
    // us at 4096^3.)
    if (rank == 0 && lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int j = 0; j < sched.n && ok; ++j) {
        const TcUnit w = tc_pair_unit(sched, j, npairs, p, nk);
        const uint32_t idesc = instr_desc(kAbType, 2 * BM, (uint32_t)w.n_w, kAT ? 1u : 0u,
                                          kBT ? 0u : 1u);
        const uint32_t b = j % kAccBufs;
        const uint32_t aph = (j / kAccBufs) & 1u;
        ok = thread_wait(smem_u32(&bars->acc_empty[b]), aph ^ 1u, p, bars, kFaultTcMmaWait);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * BN;
        for (int kt = w.kb; kt < w.ke; ++kt, ++it) {
          const uint32_t s = it % S;
          const uint32_t ph = (it / S) & 1u;
          ok = thread_wait(smem_u32(&bars->full[s]), ph, p, bars, kFaultTcMmaWait);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * kABytes);
          const uint32_t b0 = smem_u32(sB + s * kBBytes);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            const uint64_t ad = kAT ? mnmajor_desc(a0, k, kMNBlock)
                                    : kmajor_desc(a0 + (k >> 2) * kAKBlock, k & 3);
            const uint64_t bd = kBT ? kmajor_desc(b0 + (k >> 2) * kBKBlock, k & 3)
                                    : mnmajor_desc(b0, k, kMNBlock);
            mma_f16_pair(d_tmem, ad, bd, idesc, (kt > w.kb || k > 0) ? 1u : 0u);
          }
          // Both CTAs' stage s is free once these MMAs finish.
          mma_commit_pair_multicast(smem_u32(&bars->empty[s]), 0x3);
        }
        if (!ok) break;
        mma_commit_pair_multicast(smem_u32(&bars->acc_full[b]), 0x3);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int ew = warp - 2;
    unsigned char* stage0 = sEpi + ew * 2 * kEpiBufBytes;
    int nstore = 0;
    const bool with_beta = p.beta != 0.f;
    const uint32_t t_lane = tmem_base + ((uint32_t)(q * 32) << 16);
    for (int j = 0; j < sched.n; ++j) {
      const TcUnit w = tc_pair_unit(sched, j, npairs, p, nk);
      const uint32_t b = j % kAccBufs;
      const uint32_t aph = (j / kAccBufs) & 1u;
      const int row0 = w.tm * (2 * BM) + (int)rank * BM + q * 32;
      const int col0 = w.tn * BN + w.n_off;
      const T* c_in = static_cast<const T*>(p.c_in);
      const int chunks = w.n_w / kTcEpiCols;
      // A head stores its FP32 accumulator for the next pair; a tail (always
      // the pair's last unit) adds that partial to its own and finishes the
      // tile.
      const bool keep_partial = w.kind == kTcUnitHead;
      const bool finish = w.kind == kTcUnitTail;
      const bool beta_here = with_beta && !keep_partial;
      // The old C of chunk c is in old[c % 2], loaded two chunks ahead (the
      // first two while the accumulator is still being computed).
      uint4 old[2][8];
      if (beta_here) {
        load_old_row64<T>(old[0], c_in, p.ldc, p.M, p.N, row0 + lane, col0);
        if (chunks > 1)
          load_old_row64<T>(old[1], c_in, p.ldc, p.M, p.N, row0 + lane, col0 + kTcEpiCols);
      }
      if (finish) {
        // The head's partial (stored early in the other pair's share, long
        // before this last unit ends): chunk 0 into this warp's staging
        // buffers (free once its earlier stores have read them) while the
        // MMAs still run, chunks 1.. into the ring once they are done; both
        // by 16-byte cp.async, the lane-major layout giving each lane its
        // own row's values.
        int ok = 1;
        if (lane == 0) {
          ok = flag_wait_equal(partial_flag(p, w.slot, (int)rank, q), p.epoch, p.timeout_ns,
                               &bars->abort)
                   ? 1
                   : 0;
          if (!ok) {
            if (!*(volatile int*)&bars->abort) raise_fault(p.fault, kFaultTcPartialWait);
            *(volatile int*)&bars->abort = 1;
          }
          tma_store_wait_read<0>();
        }
        if (__shfl_sync(0xffffffffu, ok, 0) == 0) break;
        __threadfence();
        const float4* pb = reinterpret_cast<const float4*>(partial_block(p, w.slot, (int)rank, q));
        const uint32_t st0 = smem_u32(stage0);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          cp_async_16_cg(st0 + (jj * 32 + lane) * 16, pb + jj * 32 + lane);
        cp_async_commit();
      }
      if (!warp_wait(smem_u32(&bars->acc_full[b]), aph, p, bars, kFaultTcEpilogueWait)) break;
      tc_fence_after();
      // Ring space of this warp for partial chunks 1..3 (8 KB each): the
      // tail is the pair's last unit, so no stage is loaded any more.
      const uint32_t ring_part = smem_u32(sA) + (uint32_t)q * 3u * 8192u;
      if (finish) {
        const float4* pb = reinterpret_cast<const float4*>(partial_block(p, w.slot, (int)rank, q));
        for (int c = 1; c < chunks; ++c)
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            cp_async_16_cg(ring_part + (uint32_t)(c - 1) * 8192u + (jj * 32 + lane) * 16,
                           pb + (c * 16 + jj) * 32 + lane);
        cp_async_commit();
      }
      const uint32_t t_row = t_lane + b * BN;
#pragma unroll
      for (int c = 0; c < BN / kTcEpiCols; ++c) {
        if (c >= chunks) break;
        uint32_t r0[32], r1[32];
        tmem_ld32(t_row + c * kTcEpiCols, r0);
        tmem_ld32(t_row + c * kTcEpiCols + 32, r1);
        tmem_ld_wait(r0, r1);
        if (c == chunks - 1) {
          // This CTA's half of the accumulator is drained.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&bars->acc_empty[b]), 0));
        }
        if (keep_partial) {
          float4* dst = reinterpret_cast<float4*>(partial_block(p, w.slot, (int)rank, q)) +
                        c * 16 * 32 + lane;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const uint32_t* src = jj < 8 ? &r0[jj * 4] : &r1[(jj - 8) * 4];
            __stcg(dst + jj * 32, make_float4(__uint_as_float(src[0]), __uint_as_float(src[1]),
                                              __uint_as_float(src[2]), __uint_as_float(src[3])));
          }
          continue;
        }
        if (finish) {
          // Own sum + the head's partial, from shared memory.
          if (c == 0)
            cp_async_wait_group<1>();
          else if (c == 1)
            cp_async_wait_group<0>();
          const uint32_t src = c == 0 ? smem_u32(stage0) : ring_part + (uint32_t)(c - 1) * 8192u;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            float4 v;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                         : "r"(src + (jj * 32 + lane) * 16));
            uint32_t* d = jj < 8 ? &r0[jj * 4] : &r1[(jj - 8) * 4];
            d[0] = __float_as_uint(__uint_as_float(d[0]) + v.x);
            d[1] = __float_as_uint(__uint_as_float(d[1]) + v.y);
            d[2] = __float_as_uint(__uint_as_float(d[2]) + v.z);
            d[3] = __float_as_uint(__uint_as_float(d[3]) + v.w);
          }
          __syncwarp();   // chunk 0's staging is read before it holds output
        }
        if (p.alpha != 1.f || with_beta) scale_row64<T>(r0, r1, p.alpha, p.beta, old[c & 1]);
        if (with_beta && c + 2 < chunks)
          load_old_row64<T>(old[c & 1], c_in, p.ldc, p.M, p.N, row0 + lane,
                            col0 + (c + 2) * kTcEpiCols);
        unsigned char* buf = stage0 + (nstore & 1) * kEpiBufBytes;
        if (lane == 0) tma_store_wait_read<1>();
        __syncwarp();
        uint32_t* row = reinterpret_cast<uint32_t*>(buf + lane * 128);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint4 v;
          const uint32_t* src = ch < 4 ? &r0[ch * 8] : &r1[(ch - 4) * 8];
          v.x = pack2<T>(__uint_as_float(src[0]), __uint_as_float(src[1]));
          v.y = pack2<T>(__uint_as_float(src[2]), __uint_as_float(src[3]));
          v.z = pack2<T>(__uint_as_float(src[4]), __uint_as_float(src[5]));
          v.w = pack2<T>(__uint_as_float(src[6]), __uint_as_float(src[7]));
          *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(row) +
                                    ((ch ^ (lane & 7)) << 4)) = v;
        }
        store_tail_row(reinterpret_cast<const unsigned char*>(row), lane, p.c_out, p.ldc, p.M,
                       p.N, p.n_tma, row0 + lane, w.tn * BN + w.n_off + c * kTcEpiCols);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && p.n_tma > 0) {
          tma_store_2d(&tmC, smem_u32(buf), w.tn * BN + w.n_off + c * kTcEpiCols, row0);
          tma_store_commit();
        }
        ++nstore;
      }
      if (keep_partial) {
        // Every lane's partial is in L2 before the flag says so.
        __threadfence();
        __syncwarp();
        if (lane == 0) flag_store_release(partial_flag(p, w.slot, (int)rank, q), p.epoch);
      } else if (finish) {
        // The partial is consumed: clear the flag for the next launch (which
        // uses another epoch anyway, but may be a graph replay of this one
        // with the same epoch).
        __syncwarp();
        if (lane == 0) *partial_flag(p, w.slot, (int)rank, q) = 0u;
      }
    }
    if (lane == 0) tma_store_wait_all<0>();
    __syncwarp();
  }

  // ------------------------------------------------ teardown
  if (warp == 1 && rank == 0 && lane == 0) {
    // Every MMA of the pair has completed before TMEM is freed.
    mma_commit_pair_multicast(smem_u32(&bars->drain), 0x1);
    if (!mbar_wait_bounded(smem_u32(&bars->drain), 0, p.timeout_ns, nullptr))
      raise_fault(p.fault, kFaultDrainWait);
  }
  if (warp == 0 && lane == 0 && rank == 0 && bars->abort) {
    // Let in-flight loads (both CTAs count on the even CTA's barriers) land.
    const uint32_t first = issued > (uint32_t)S ? issued - S : 0;
    for (uint32_t it = first; it < issued; ++it) {
      if (!mbar_wait_bounded(smem_u32(&bars->full[it % S]), (it / S) & 1u, p.timeout_ns,
                             nullptr)) {
        raise_fault(p.fault, kFaultDrainWait);
        break;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();     // neither CTA leaves while the pair may still touch its memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <typename T, uint32_t kAb, bool kAT, bool kBT>
cudaError_t launch_typed(const TcParams& p, const CUtensorMap* tmA, const CUtensorMap* tmB,
                         const CUtensorMap* tmC, int pairs, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_pair_kernel<T, kAb, kAT, kBT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kTc2SmemBytes);
  if (e != cudaSuccess) return e;
  return launch_gemm_kernel(gemm_tc_pair_kernel<T, kAb, kAT, kBT>, dim3(2 * pairs),
                            dim3(kTcThreads), kTc2SmemBytes, stream, *tmA, *tmB, *tmC, p);
}

template <typename T, uint32_t kAb>
cudaError_t launch_ops(const TcParams& p, const CUtensorMap* tmA, const CUtensorMap* tmB,
                       const CUtensorMap* tmC, int pairs, cudaStream_t stream) {
  if (p.op_a && p.op_b) return launch_typed<T, kAb, true, true>(p, tmA, tmB, tmC, pairs, stream);
  if (p.op_a) return launch_typed<T, kAb, true, false>(p, tmA, tmB, tmC, pairs, stream);
  if (p.op_b) return launch_typed<T, kAb, false, true>(p, tmA, tmB, tmC, pairs, stream);
  return launch_typed<T, kAb, false, false>(p, tmA, tmB, tmC, pairs, stream);
}

}  // namespace

static_assert(sizeof(Barriers) <= 256, "barrier block must fit its reserved space");

int tc_pair_resident_clusters() {
  // Every instance has the same block size and shared memory, so one
  // stands for all.
  const auto kernel = gemm_tc_pair_kernel<__half, 0, false, false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTc2SmemBytes) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTc2SmemBytes;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return clusters;
}

cudaError_t launch_gemm_tc_pair(int dtype, const TcParams& p, const CUtensorMap* tmA,
                                const CUtensorMap* tmB, const CUtensorMap* tmC, int pairs,
                                cudaStream_t stream) {
  if (dtype == 1) return launch_ops<__half, 0>(p, tmA, tmB, tmC, pairs, stream);
  return launch_ops<__nv_bfloat16, 1>(p, tmA, tmB, tmC, pairs, stream);
}

}  // namespace dgemm
