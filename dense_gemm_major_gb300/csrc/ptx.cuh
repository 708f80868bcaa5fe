// Inline-PTX helpers for sm_103a: shared-memory addresses, mbarriers, TMA
// (cp.async.bulk.tensor), cp.async with zero fill, and bounded waits.
//
// Every wait in this library is bounded: a wait that has not completed after
// `timeout_ns` of %globaltimer time gives up and reports failure to its
// caller, which records a fault code in the library's device fault word and
// unwinds the kernel instead of spinning for ever.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace dgemm {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// `raw` (a __shared__ array) advanced to the next 1024-byte boundary of the
// shared window.  The pointer is formed by indexing the array itself, so the
// compiler keeps it in the shared address space and emits shared loads and
// stores through it (a pointer rounded through an integer becomes generic:
// on sm_103a a generic 16-byte load from shared memory was measured at 4
// wavefronts where the same ld.shared takes 2).
__device__ __forceinline__ unsigned char* align_smem_1024(unsigned char* raw) {
  const uint32_t pad = (1024u - (smem_u32(raw) & 1023u)) & 1023u;
  return raw + pad;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but a thread whose phase is not complete yet is
// suspended in hardware until it completes or about `hint_ns` pass, instead
// of returning at once: a waiting warp issues almost nothing while it waits.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity,
                                                      uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false if
// `timeout_ns` elapses first, or if `*abort` becomes non-zero (another role
// of the same CTA gave up).  Each try suspends the thread for up to 10 us, so
// the timeout and the abort flag are checked at least every few ms.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t timeout_ns,
                                                  const volatile int* abort) {
  constexpr uint32_t kSuspendNs = 10000;
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_suspend(bar, parity, kSuspendNs)) return true;
    if ((it & 255u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
  }
}

// As mbar_wait_bounded, but every try is a plain try_wait (no suspend-time
// hint), for the latency-critical waits of the TMA producer and the MMA
// issuer: a thread that was suspended resumes later than the phase
// completes (measured: 4096^3 FP16 on CTA pairs 94.2 -> 92.2 us).
__device__ __forceinline__ bool mbar_wait_spin_bounded(uint32_t bar, uint32_t parity,
                                                       uint64_t timeout_ns,
                                                       const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 1023u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
  }
}

// Release store / acquire poll of a 32-bit flag in global memory, for
// handing a partial result from one CTA to another of the same grid.
__device__ __forceinline__ void flag_store_release(unsigned* f, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned flag_load_acquire(const unsigned* f) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
  return v;
}
// Waits until *f == v.  Returns false if `timeout_ns` elapses first or
// `*abort` becomes non-zero.
__device__ __forceinline__ bool flag_wait_equal(const unsigned* f, unsigned v, uint64_t timeout_ns,
                                                const volatile int* abort) {
  if (flag_load_acquire(f) == v) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (flag_load_acquire(f) == v) return true;
    if ((it & 63u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
  }
}

// ---------------------------------------------------------------- clusters

// Shared::cluster address of the object at shared offset `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// All threads of every CTA of the cluster: release this CTA's earlier
// memory operations, acquire the others'.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16-byte store to the shared memory of a CTA of the cluster (address from
// mapa_shared).
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// ---------------------------------------------------------------- dependent launch

// Programmatic dependent launch: a kernel launched with the
// programmatic-stream-serialization attribute may start (run its prologue)
// while the kernel before it in the stream is still running.
// wait_prior_grids blocks until that kernel has completed and its memory
// operations are visible (a no-op without the attribute): every global
// memory access of the kernel comes after it.  allow_dependent_grids lets
// the next kernel, if launched the same way, be scheduled as SMs free up;
// it still waits for this kernel's completion before touching memory.
__device__ __forceinline__ void wait_prior_grids() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependent_grids() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* desc) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(desc)) : "memory");
}

// 2-D tiled load global -> shared; completion is signalled on `bar` as
// transaction bytes.  x is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* desc, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(desc)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// L2 cache hints on the operand loads, a compile-time switch for the
// access-policy measurement (the GB300 GEMM roadmap, section 3.2, suggests
// keeping reused data resident in L2; its section 6.1 warns that marking
// data read once does the opposite).  DENSE_GEMM_L2_HINT: 0 (the default)
// plain loads; 1 A evict-first, B evict-last; 2 A evict-last, B
// evict-first.  Build with -DDENSE_GEMM_L2_HINT=n in DENSE_GEMM_NVCC_FLAGS.
#ifndef DENSE_GEMM_L2_HINT
#define DENSE_GEMM_L2_HINT 0
#endif

__device__ __forceinline__ uint64_t l2_policy(bool evict_first) {
  uint64_t p;
  if (evict_first)
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  else
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// tma_load_2d with an L2 cache-policy operand.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* desc,
                                                 uint32_t bar, int32_t x, int32_t y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(desc)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// The load of operand kOperand (0 = A, 1 = B) under DENSE_GEMM_L2_HINT.
template <int kOperand>
__device__ __forceinline__ void tma_load_operand(uint32_t dst, const CUtensorMap* desc,
                                                 uint32_t bar, int32_t x, int32_t y) {
#if DENSE_GEMM_L2_HINT == 0
  tma_load_2d(dst, desc, bar, x, y);
#else
  tma_load_2d_hint(dst, desc, bar, x, y, l2_policy((DENSE_GEMM_L2_HINT == 1) == (kOperand == 0)));
#endif
}

// 2-D tiled store shared -> global (out-of-range rows/columns are clipped).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* desc, uint32_t src, int32_t x,
                                             int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(desc)),
      "r"(src), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_store_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until at most N committed store groups still read shared memory.
template <int N>
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- cp.async

// 4-byte copy global -> shared; when `valid` is false nothing is read and
// the destination is zero-filled.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}

// Arrives on `bar` once all of this thread's earlier cp.async copies have
// landed; the barrier's expected count includes this arrival.
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// 16-byte cp.async global -> shared through L2 only (data another SM just
// wrote), completed by commit / wait_group.
__device__ __forceinline__ void cp_async_16_cg(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---------------------------------------------------------------- faults

// Fault codes OR-ed into the library's device fault word.
enum FaultCode : unsigned {
  kFaultSgemmFullWait = 1u << 0,
  kFaultTcProducerWait = 1u << 1,
  kFaultTcMmaWait = 1u << 2,
  kFaultTcEpilogueWait = 1u << 3,
  kFaultSelftestWait = 1u << 4,
  kFaultDrainWait = 1u << 5,
  kFaultTcPairTmem = 1u << 6,   // the two CTAs of a pair got different TMEM bases
  kFaultTcPartialWait = 1u << 7,   // a K-split piece's partial never arrived
  kFaultSgemmPieceWait = 1u << 8,  // an SGEMM stream-K piece's partner never published
};

__device__ __forceinline__ void raise_fault(unsigned* fault, unsigned code) {
  if (fault != nullptr) atomicOr(fault, code);
}

}  // namespace dgemm
