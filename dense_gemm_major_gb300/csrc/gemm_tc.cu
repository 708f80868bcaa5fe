// FP16 / BF16 GEMM on sm_103a tensor cores: C = A . B, row-major, FP32
// accumulation in tensor memory, FP16 / BF16 output rounded to nearest-even.
//
// The structure is the five-step flow of the GB300 GEMM roadmap (m.nxbn.cn,
// section 4.2): TMA copies A and B tiles into shared memory; tcgen05.mma reads
// them from shared memory and accumulates into tensor memory (TMEM); loading
// of the next tiles continues meanwhile; after the K loop tcgen05.ld brings
// the accumulator into registers; the epilogue writes C to global memory.
// Section 4.1 of the same page: the MMA is issued asynchronously and the
// issuing warp does not wait for it; section 3.1: a 3-4 stage shared-memory
// ring overlaps loads with MMAs; section 1.1: the data supply, not the MMA
// unit, is what limits a GEMM on this chip.
//
// GB300-specific choices (no page gives a tcgen05 kernel):
//  * Persistent grid, at most one CTA per SM, static round-robin over
//    128 x 256 output tiles in groups of 8 tile rows (L2 reuse).  The tiles
//    of a last partial round run as 2 or 4 column parts (N = 128 or 64 per
//    tcgen05.mma, full K each), so that round ends sooner without any
//    cross-CTA reduction: results are the same bits as unsplit tiles.
//  * Warp roles: warp 0 = TMA producer, warp 1 = TMEM allocator and MMA
//    issuer (one thread issues every tcgen05.mma), warps 2-5 = epilogue (each
//    owns the 32 TMEM lanes its warp index mod 4 may access).
//  * Ring: 4 stages of A (128 x 64, K-major, 128-byte swizzle) and B (64 x 256,
//    N-major, as four 64-column boxes, 128-byte swizzle); `full` mbarriers
//    carry TMA transaction bytes, `empty` mbarriers are arrived by
//    tcgen05.commit once the MMAs reading a stage are done.
//  * Accumulator: two 128 x 256 FP32 buffers in TMEM (all 512 columns), so
//    the epilogue of one tile overlaps the main loop of the next.
//  * Epilogue: tcgen05.ld 32x32b -> FP32 registers -> RN conversion ->
//    128-byte-swizzled shared staging (conflict-free) -> TMA store of 32 x 64
//    boxes; TMA clips rows and columns beyond M and N.
//  * Every mbarrier wait is bounded; a wait that gives up records a fault,
//    stops this CTA's roles, drains its copies and MMAs and frees TMEM.
//  * Operands stored transposed (kAT: A stored K x M; kBT: B stored N x K,
//    the column-major B of the m.lqnn.cn SGEMM article, section 3.1) need no
//    copy: TMA reads them as stored and tcgen05.mma takes an MN-major A and
//    a K-major B directly; only the TMA coordinates, the shared-memory
//    descriptors and the instruction descriptor's major bits change.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "launch.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace dgemm {
namespace {

constexpr int BM = kTcBM;
constexpr int BN = kTcBN;
constexpr int BK = kTcBK;
constexpr int S = kTcStages;
constexpr int UMMA_K = 16;                         // K per tcgen05.mma (16-bit inputs)
constexpr uint32_t kABytes = BM * BK * 2;          // 16 KB
constexpr uint32_t kBBoxBytes = 64 * BK * 2;       // one 64-column box of B: 8 KB
constexpr uint32_t kBBytes = BN * BK * 2;          // 32 KB
constexpr uint32_t kEpiBufBytes = 32 * kTcEpiCols * 2;   // 4 KB
constexpr uint32_t kTmemCols = 2 * BN;             // two accumulators
constexpr int kEpiWarps = 4;

static_assert(BK * 2 == 128, "A rows of a stage are one 128-byte swizzle row");
static_assert(kTcEpiCols * 2 == 128, "epilogue boxes are one 128-byte swizzle row wide");
static_assert(kTmemCols == 512, "TMEM holds exactly two accumulators");

struct alignas(8) Barriers {
  uint64_t full[S];
  uint64_t empty[S];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Work unit u of the persistent grid: output tile (tm, tn) in grouped raster
// order, the columns [n_off, n_off + n_w) of it that the unit computes (the
// whole 256 columns, or one of 2 or 4 parts of a split tile), and its k-tile
// range [kb, ke) (a k-slice in split-K mode, else all of K).
struct Unit {
  int tm, tn, n_off, n_w, kb, ke, slice;
};
__device__ __forceinline__ Unit unit_of(int u, const TcParams& p, int nk) {
  Unit w;
  int tile;
  w.kb = 0;
  w.ke = nk;
  w.slice = -1;
  w.n_off = 0;
  w.n_w = BN;
  if (p.slices > 1) {
    tile = u / p.slices;
    w.slice = u - tile * p.slices;
    w.kb = w.slice * nk / p.slices;
    w.ke = (w.slice + 1) * nk / p.slices;
  } else if (u < p.full_tiles) {
    tile = u;
  } else {
    const int j = u - p.full_tiles;
    const int part = j % p.parts;
    tile = p.full_tiles + j / p.parts;
    w.n_w = BN / p.parts;
    w.n_off = part * w.n_w;
  }
  grouped_tile(tile, p.tiles_m, p.tiles_n, p.group_m, w.tm, w.tn);
  return w;
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

// Warp-uniform bounded wait: lane 0 polls, the result is broadcast.
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
      // Only the role that timed out raises its code; roles that stop
      // because another one gave up just follow.
      if (!*(volatile int*)&bars->abort) raise_fault(p.fault, fault_code);
      *(volatile int*)&bars->abort = 1;
    }
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <typename T, uint32_t kAbType, bool kAT, bool kBT>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* const base = align_smem_1024(smem_raw);
  unsigned char* sA = base;
  unsigned char* sB = sA + S * kABytes;
  unsigned char* sEpi = sB + S * kBBytes;
  Barriers* bars = reinterpret_cast<Barriers*>(sEpi + kEpiWarps * 2 * kEpiBufBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_units = p.slices > 1 ? p.tiles_m * p.tiles_n * p.slices
                                     : p.full_tiles + p.split_tiles * p.parts;
  const int nk = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars->acc_full[b]), 1);
      mbar_init(smem_u32(&bars->acc_empty[b]), kEpiWarps);
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
  if (warp == 1) tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;
  wait_prior_grids();
  allow_dependent_grids();

  uint32_t issued = 0;   // producer: k-tiles issued (lane 0 of warp 0)

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const Unit w = unit_of(u, p, nk);
      const int tm = w.tm, tn = w.tn;
      const int boxes = w.n_w / 64;   // B boxes (64 columns each) this unit needs
      for (int kt = w.kb; kt < w.ke; ++kt, ++it) {
        const uint32_t s = it % S;
        const uint32_t ph = (it / S) & 1u;
        ok = warp_wait(smem_u32(&bars->empty[s]), ph ^ 1u, p, bars, kFaultTcProducerWait);
        if (!ok) break;
        if (lane == 0) {
          const uint32_t fb = smem_u32(&bars->full[s]);
          mbar_arrive_expect_tx(fb, kABytes + boxes * kBBoxBytes);
          const uint32_t adst = smem_u32(sA + s * kABytes);
          if constexpr (!kAT) {
            tma_load_operand<0>(adst, &tmA, fb, kt * BK, tm * BM);
          } else {   // A stored K x M: two 64-row (m) blocks, MN-major
            for (int j = 0; j < BM / 64; ++j)
              tma_load_operand<0>(adst + j * kBBoxBytes, &tmA, fb, tm * BM + j * 64, kt * BK);
          }
          const uint32_t bdst = smem_u32(sB + s * kBBytes);
          for (int j = 0; j < boxes; ++j) {
            const int n = tn * BN + w.n_off + j * 64;
            if constexpr (!kBT)
              tma_load_operand<1>(bdst + j * kBBoxBytes, &tmB, fb, n, kt * BK);
            else   // B stored N x K: 64 rows (n) of 64 k each, K-major
              tma_load_operand<1>(bdst + j * kBBoxBytes, &tmB, fb, kt * BK, n);
          }
          issued = it + 1;
        }
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    // One thread waits and issues, with no warp-wide synchronisation between
    // stages (as in the pair kernel, where that bookkeeping had left the
    // tensor pipe idle for part of every stage).
    if (lane == 0) {
      uint32_t it = 0;
      int local = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x, ++local) {
        const Unit w = unit_of(u, p, nk);
        const uint32_t idesc = instr_desc(kAbType, BM, (uint32_t)w.n_w, kAT ? 1u : 0u,
                                          kBT ? 0u : 1u);
        const uint32_t b = local & 1;
        const uint32_t aph = (local >> 1) & 1u;
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
            // A K-major (MN-major when stored transposed), B MN-major
            // (K-major when stored transposed).
            const uint64_t ad = kAT ? mnmajor_desc(a0, k) : kmajor_desc(a0, k);
            const uint64_t bd = kBT ? kmajor_desc(b0, k) : mnmajor_desc(b0, k);
            mma_f16(d_tmem, ad, bd, idesc, (kt > w.kb || k > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&bars->empty[s]));   // frees the stage when the MMAs finish
        }
        if (!ok) break;
        mma_commit(smem_u32(&bars->acc_full[b]));   // accumulator ready
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue
    const int q = warp & 3;                    // TMEM lane quadrant of this warp
    const int ew = warp - 2;                   // epilogue warp index 0..3
    unsigned char* stage0 = sEpi + ew * 2 * kEpiBufBytes;
    int local = 0;
    int nstore = 0;
    const bool with_beta = p.beta != 0.f;
    // Rounds 64 FP32 columns (r0: 32, r1: the next 32) of this lane's row to
    // T, stages them 128-byte swizzled and TMA-stores the warp's 32 x 64 box
    // at tile column `col`.
    auto store_box = [&](const uint32_t (&r0)[32], const uint32_t (&r1)[32], int tm, int tn,
                         int col) {
      unsigned char* buf = stage0 + (nstore & 1) * kEpiBufBytes;
      // The store issued from this buffer two boxes ago must have read it.
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
      store_tail_row(reinterpret_cast<const unsigned char*>(row), lane, p.c_out, p.ldc, p.M, p.N,
                     p.n_tma, tm * BM + q * 32 + lane, tn * BN + col);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && p.n_tma > 0) {
        tma_store_2d(&tmC, smem_u32(buf), tn * BN + col, tm * BM + q * 32);
        tma_store_commit();
      }
      ++nstore;
    };
    for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++local) {
      const Unit w = unit_of(u, p, nk);
      const uint32_t b = local & 1;
      const uint32_t aph = (local >> 1) & 1u;
      const int grow = w.tm * BM + q * 32 + lane;
      const int col0 = w.tn * BN + w.n_off;
      const T* c_in = static_cast<const T*>(p.c_in);
      // (Split-K slices leave alpha and beta to the reduction.)
      const bool old_needed = with_beta && w.slice < 0;
      const int chunks = w.n_w / kTcEpiCols;
      // The old C of chunk c is in old[c % 2], loaded two chunks ahead (the
      // first two while the accumulator is still being computed).
      uint4 old[2][8];
      if (old_needed) {
        load_old_row64<T>(old[0], c_in, p.ldc, p.M, p.N, grow, col0);
        if (chunks > 1)
          load_old_row64<T>(old[1], c_in, p.ldc, p.M, p.N, grow, col0 + kTcEpiCols);
      }
      if (!warp_wait(smem_u32(&bars->acc_full[b]), aph, p, bars, kFaultTcEpilogueWait)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + b * BN;
#pragma unroll
      for (int c = 0; c < BN / kTcEpiCols; ++c) {
        if (c >= chunks) break;
        uint32_t r0[32], r1[32];
        tmem_ld32(t_row + c * kTcEpiCols, r0);
        tmem_ld32(t_row + c * kTcEpiCols + 32, r1);
        tmem_ld_wait(r0, r1);
        if (c == chunks - 1) {
          // The accumulator buffer is free for the next unit's MMAs.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty[b]));
        }
        if (w.slice < 0) {
          if (p.alpha != 1.f || with_beta)
            scale_row64<T>(r0, r1, p.alpha, p.beta, old[c & 1]);
          if (old_needed && c + 2 < chunks)
            load_old_row64<T>(old[c & 1], c_in, p.ldc, p.M, p.N, grow,
                              col0 + (c + 2) * kTcEpiCols);
          store_box(r0, r1, w.tm, w.tn, w.n_off + c * kTcEpiCols);
        } else {
          // Split-K: this lane's row of the FP32 partial, columns beyond the
          // workspace width (ldw >= N, a multiple of 4) left out.
          const int gcol = w.tn * BN + c * kTcEpiCols;
          if (grow < p.M) {
            float* dst = p.ws + (long long)w.slice * p.M * p.ldw + (long long)grow * p.ldw + gcol;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (gcol + 4 * j + 3 < p.ldw) {
                const uint32_t* src = j < 8 ? &r0[j * 4] : &r1[(j - 8) * 4];
                *reinterpret_cast<uint4*>(dst + 4 * j) = make_uint4(src[0], src[1], src[2], src[3]);
              }
            }
          }
        }
      }
    }
    if (lane == 0) tma_store_wait_all<0>();
    __syncwarp();
  }

  // ------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && bars->abort) {
    // Let this CTA's in-flight TMA loads land before the CTA exits.
    const uint32_t first = issued > (uint32_t)S ? issued - S : 0;
    for (uint32_t it = first; it < issued; ++it) {
      if (!mbar_wait_bounded(smem_u32(&bars->full[it % S]), (it / S) & 1u, p.timeout_ns,
                             nullptr)) {
        raise_fault(p.fault, kFaultDrainWait);
        break;
      }
    }
  }
  if (warp == 1) {
    tc_fence_after();
    if (lane == 0) {
      // Wait for every MMA this CTA issued before freeing TMEM.
      mma_commit(smem_u32(&bars->drain));
      if (!mbar_wait_bounded(smem_u32(&bars->drain), 0, p.timeout_ns, nullptr))
        raise_fault(p.fault, kFaultDrainWait);
    }
    __syncwarp();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <typename T, uint32_t kAb, bool kAT, bool kBT>
cudaError_t launch_typed(const TcParams& p, const CUtensorMap* tmA, const CUtensorMap* tmB,
                         const CUtensorMap* tmC, int grid, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<T, kAb, kAT, kBT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_gemm_kernel(gemm_tc_kernel<T, kAb, kAT, kBT>, dim3(grid), dim3(kTcThreads),
                            kTcSmemBytes, stream, *tmA, *tmB, *tmC, p);
}

template <typename T, uint32_t kAb>
cudaError_t launch_ops(const TcParams& p, const CUtensorMap* tmA, const CUtensorMap* tmB,
                       const CUtensorMap* tmC, int grid, cudaStream_t stream) {
  if (p.op_a && p.op_b) return launch_typed<T, kAb, true, true>(p, tmA, tmB, tmC, grid, stream);
  if (p.op_a) return launch_typed<T, kAb, true, false>(p, tmA, tmB, tmC, grid, stream);
  if (p.op_b) return launch_typed<T, kAb, false, true>(p, tmA, tmB, tmC, grid, stream);
  return launch_typed<T, kAb, false, false>(p, tmA, tmB, tmC, grid, stream);
}

}  // namespace

static_assert(sizeof(Barriers) <= 256, "barrier block must fit its reserved space");

cudaError_t launch_gemm_tc(int dtype, const TcParams& p, const CUtensorMap* tmA,
                           const CUtensorMap* tmB, const CUtensorMap* tmC, int grid,
                           cudaStream_t stream) {
  if (dtype == 1) return launch_ops<__half, 0>(p, tmA, tmB, tmC, grid, stream);
  return launch_ops<__nv_bfloat16, 1>(p, tmA, tmB, tmC, grid, stream);
}

}  // namespace dgemm
