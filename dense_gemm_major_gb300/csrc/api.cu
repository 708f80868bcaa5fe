// C-ABI entry points: argument validation, path selection, TMA descriptor
// encoding and launch.  See include/dense_gemm.h for the contract.
//
// The dispatcher plays the role of the pages' torch-extension binding macros
// ("[CUDA 优化实战] sgemm - 超越 cuBLAS", section 1 binding_func_gen and section 2
// binding_tiled_func_gen: read M, K, N, pick grid and block, launch on the
// caller's stream), with plain pointers and sizes instead of tensors, and a
// shape/alignment-driven choice of kernel path in the spirit of the library
// launcher described in the GB300 GEMM roadmap (m.nxbn.cn, section 1.2).
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "dense_gemm.h"
#include "launch.h"
#include "ptx.cuh"

namespace {

// The device fault word: kernels OR a dgemm::FaultCode into it when a
// bounded wait gives up.  One copy per device.
__device__ unsigned g_fault_word;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool probed = false;
  bool supported = false;
  int sms = 0;
  // 2-CTA clusters of the pair kernel that fit on the device at once
  // (cudaOccupancyMaxActiveClusters; 0 if the query failed).
  int pair_clusters = 0;
  // Clusters of the SGEMM kernel over K that fit at once (the same query).
  dgemm::SgemmClusterCaps sgemm_caps{};
  unsigned* fault = nullptr;  // device address of g_fault_word
};

std::mutex g_mu;
DeviceInfo g_devices[kMaxDevices];

// Device workspaces: one per (device, stream, use), grown on demand, never
// shrunk, freed at process exit by the driver.  Use kWsPartials holds
// split-K slices or stream-K partial tiles, kWsPack a packed operand; one
// call can need both.
struct Workspace {
  float* ptr = nullptr;
  size_t bytes = 0;
  unsigned epoch = 0;   // kWsFlags: the last epoch handed to a launch
};
// kWsFlags holds the hand-over flags of cut tiles (the pair kernel's K
// split, the SGEMM's stream-K pieces): zeroed when (re)allocated, then only
// ever set to a launch's epoch (or cleared).
constexpr int kWsPartials = 0, kWsPack = 1, kWsFlags = 2;
std::map<std::tuple<int, cudaStream_t, int>, Workspace> g_workspaces;   // guarded by g_mu

gemm_status_t get_workspace(cudaStream_t stream, size_t bytes, float** out,
                            int use = kWsPartials) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_UNSUPPORTED_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace& w = g_workspaces[std::make_tuple(dev, stream, use)];
  if (w.bytes < bytes) {
    // Earlier work queued on this stream may still use the old buffer.
    if (w.ptr != nullptr) {
      if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
      }
      cudaFree(w.ptr);
      w.ptr = nullptr;
      w.bytes = 0;
    }
    if (cudaMalloc(&w.ptr, bytes) != cudaSuccess) {
      cudaGetLastError();
      w.ptr = nullptr;
      return GEMM_ERR_LAUNCH;
    }
    w.bytes = bytes;
    if (use == kWsFlags && cudaMemsetAsync(w.ptr, 0, bytes, stream) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_LAUNCH;
    }
  }
  *out = w.ptr;
  return GEMM_OK;
}

// The next epoch of the K-split flags of (current device, stream); never 0.
unsigned next_epoch(cudaStream_t stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) cudaGetLastError();
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace& w = g_workspaces[std::make_tuple(dev, stream, kWsFlags)];
  if (++w.epoch == 0) w.epoch = 1;
  return w.epoch;
}

constexpr long long kSplitkWorkspaceCap = 64ll << 20;   // bytes

// Packing a transposed FP32 operand (see plan_impl): minimum reuse of each
// packed element, minimum M * N * K, and the largest scratch copy.
constexpr int kPackMinReuse = 256;
constexpr long long kPackMinWork = 1ll << 30;
constexpr long long kPackCapBytes = 1ll << 30;
// Re-pitching row-major FP32 operands whose base or leading dimension is not
// 16-byte aligned (so that TMA can stage them): minimum M * N * K.
constexpr long long kRepitchMinWork = 1ll << 29;

inline long long round4(long long x) { return (x + 3) / 4 * 4; }

// FP32 split-K slice count: the s in [2, min(nk, 32)] that minimises
// ceil(tiles * s / sms) * (nk / s + kSgemmSliceCost), the k-tiles on the
// busiest SM (two co-resident CTAs share its FMA pipe, so they count twice)
// plus a fixed cost per slice (pipeline fill, partial store, reduction)
// worth kSgemmSliceCost k-tiles; the smallest such s; then bounded so the
// workspace stays under the cap.  Measured on GB300 (us, s = 2/4/8/16):
// 256^3 23.2/17.1/15.0/-, 384^3 29.3/21.2/19.1/17.0 (12), 512^3
// 33.4/25.3/21.1/21.1, 768^3 47.7/31.4/33.4/41.6, 256 x 256 x 1024
// 55.9/33.4/23.2/21.1; the rule picks 8, 12, 9, 4 and 32.
constexpr double kSgemmSliceCost = 2.0;
int sgemm_splitk_slices(int tiles, int sms, int nk, int M, int N) {
  if (tiles <= 0 || sms <= 0) return 1;
  const int smax = nk < 32 ? nk : 32;
  int best = 1;
  double best_cost = 0.0;
  for (int s = 2; s <= smax; ++s) {
    const double waves = (double)(((long long)tiles * s + sms - 1) / sms);
    const double cost = waves * ((double)nk / s + kSgemmSliceCost);
    if (best == 1 || cost < best_cost - 1e-9) {
      best = s;
      best_cost = cost;
    }
  }
  const long long slice_bytes = (long long)M * (((long long)N + 3) / 4 * 4) * 4;
  while (best > 1 && best * slice_bytes > kSplitkWorkspaceCap) --best;
  return best >= 2 ? best : 1;
}

// Slices for a split-K problem, bounded so the workspace stays under the cap.
int splitk_slices_capped(int tiles, int slots, int nk, int M, int N) {
  int s = dgemm::splitk_slices(tiles, slots, nk);
  const long long slice_bytes = (long long)M * (((long long)N + 3) / 4 * 4) * 4;
  while (s > 1 && s * slice_bytes > kSplitkWorkspaceCap) --s;
  return s >= 2 ? s : 1;
}

unsigned long long wait_timeout_ns() {
  static const unsigned long long v = [] {
    unsigned long long ms = 2000;  // a bounded wait gives up after 2 s by default
    if (const char* s = std::getenv("DENSE_GEMM_TIMEOUT_MS")) {
      char* end = nullptr;
      const unsigned long long x = std::strtoull(s, &end, 10);
      if (end != s && x > 0) ms = x;
    }
    return ms * 1000000ull;
  }();
  return v;
}

gemm_status_t current_device(DeviceInfo** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GEMM_ERR_UNSUPPORTED_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_devices[dev];
  if (!d.probed) {
    d.probed = true;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    // The kernels are built for sm_103a only.
    d.supported = (prop.major == 10 && prop.minor == 3);
    d.sms = prop.multiProcessorCount;
    void* addr = nullptr;
    if (d.supported && cudaGetSymbolAddress(&addr, g_fault_word) != cudaSuccess) {
      cudaGetLastError();
      d.supported = false;
    }
    d.fault = static_cast<unsigned*>(addr);
    if (d.supported) {
      d.pair_clusters = dgemm::tc_pair_resident_clusters();
      d.sgemm_caps = dgemm::sgemm_cluster_caps();
    }
  }
  if (!d.supported) return GEMM_ERR_UNSUPPORTED_DEVICE;
  *out = &d;
  return GEMM_OK;
}

// cuTensorMapEncodeTiled, fetched from the driver once.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      p = nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// 2-D row-major tensor {inner, outer} with row pitch `pitch_bytes`.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
               uint64_t outer, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {pitch_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bytes spanned by a rows x cols block with leading dimension ld.
inline uint64_t span_bytes(long long rows, long long cols, long long ld, int es) {
  if (rows <= 0 || cols <= 0) return 0;
  return (uint64_t)((rows - 1) * ld + cols) * (uint64_t)es;
}

inline bool overlap(const void* a, uint64_t an, const void* b, uint64_t bn) {
  if (an == 0 || bn == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Measurement override: DENSE_GEMM_SGEMM_PACK=0 never packs a transposed
// FP32 operand, =1 packs one whatever the reuse (-1 = no override).
int forced_sgemm_pack() {
  static const int v = [] {
    const char* s = std::getenv("DENSE_GEMM_SGEMM_PACK");
    if (s == nullptr) return -1;
    if (std::strcmp(s, "0") == 0) return 0;
    if (std::strcmp(s, "1") == 0) return 1;
    return -1;
  }();
  return v;
}

// Measurement override: DENSE_GEMM_SGEMM_REPITCH=0 never re-pitches an
// unaligned row-major FP32 operand, =1 always does (-1 = no override).
int forced_sgemm_repitch() {
  static const int v = [] {
    const char* s = std::getenv("DENSE_GEMM_SGEMM_REPITCH");
    if (s == nullptr) return -1;
    if (std::strcmp(s, "0") == 0) return 0;
    if (std::strcmp(s, "1") == 0) return 1;
    return -1;
  }();
  return v;
}

// Measurement override: DENSE_GEMM_TC_STREAMK=0 turns off the pair kernel's
// stream-K share (its last partial round then runs as column parts, or as
// it is).
bool tc_streamk_disabled() {
  static const bool v = [] {
    const char* s = std::getenv("DENSE_GEMM_TC_STREAMK");
    return s != nullptr && std::strcmp(s, "0") == 0;
  }();
  return v;
}

// Measurement override: DENSE_GEMM_TC_SK_ROUNDS=2 makes the pair kernel's
// stream-K share cover the last partial round and the two before it
// whenever there are that many.
int tc_sk_min_rounds() {
  static const int v = [] {
    const char* s = std::getenv("DENSE_GEMM_TC_SK_ROUNDS");
    return s != nullptr && std::strcmp(s, "2") == 0 ? 2 : 1;
  }();
  return v;
}

// Measurement override: DENSE_GEMM_TC_SPLIT=0 turns off the column split of
// the last partial round of FP16/BF16 tiles.
bool tc_split_disabled() {
  static const bool v = [] {
    const char* s = std::getenv("DENSE_GEMM_TC_SPLIT");
    return s != nullptr && std::strcmp(s, "0") == 0;
  }();
  return v;
}

// Measurement override: DENSE_GEMM_TC_GROUP=<n> sets the FP16/BF16 tile rows
// per rasterisation group (0 = default).
int tc_group_override() {
  static const int v = [] {
    const char* s = std::getenv("DENSE_GEMM_TC_GROUP");
    return s != nullptr ? std::atoi(s) : 0;
  }();
  return v;
}

// Measurement override: DENSE_GEMM_TC_KERNEL=single|pair forces the FP16/BF16
// kernel (0 = no override, 1 = single CTAs, 2 = CTA pairs).
int forced_tc_kernel() {
  static const int v = [] {
    const char* s = std::getenv("DENSE_GEMM_TC_KERNEL");
    if (s == nullptr) return 0;
    if (std::strcmp(s, "single") == 0) return 1;
    if (std::strcmp(s, "pair") == 0) return 2;
    return 0;
  }();
  return v;
}

// Measurement override: DENSE_GEMM_SGEMM_SLICES=s (2..32) runs every FP32
// product as split-K with s slices (capped at one k-tile per slice); 0 = no
// override.
int forced_sgemm_slices() {
  static const int v = [] {
    const char* s = std::getenv("DENSE_GEMM_SGEMM_SLICES");
    if (s == nullptr) return 0;
    const int x = std::atoi(s);
    return x >= 2 && x <= 32 ? x : 0;
  }();
  return v;
}

// Measurement override: DENSE_GEMM_SGEMM_CLUSTER=0 runs the FP32 grid of
// two CTAs per tile as stream-K pieces meeting through flags instead of
// 2-CTA clusters.
bool sgemm_clusters_off() {
  static const bool v = [] {
    const char* s = std::getenv("DENSE_GEMM_SGEMM_CLUSTER");
    return s != nullptr && std::strcmp(s, "0") == 0;
  }();
  return v;
}

// Measurement override: DENSE_GEMM_SGEMM_TILE=narrow|wide forces the FP32
// tile configuration (0 = no override).
int forced_sgemm_tn() {
  static const int v = [] {
    const char* s = std::getenv("DENSE_GEMM_SGEMM_TILE");
    if (s == nullptr) return 0;
    if (std::strcmp(s, "narrow") == 0) return 8;
    if (std::strcmp(s, "wide") == 0) return 16;
    if (std::strcmp(s, "narrow1") == 0) return 9;
    return 0;
  }();
  return v;
}

// FP32 tile configuration of a grid that is not split-K: 16 = wide (8 x 16
// per thread, one CTA per SM), 9 = narrow with one CTA per SM, 8 = narrow
// with two.  Picks the largest (speed relative to wide) x (share of the CTA
// slots busy): a grid of more tiles than slots is balanced by stream-K
// (share 1), a smaller one fills tiles / slots (twice that when it runs as
// two k-halves per tile).  Relative speeds measured on GB300 at 4096^3,
// 8192 x 8192 x 4096 and 6144 x 6144 x 2048: wide 1.00, narrow/1 0.93,
// narrow/2 0.92.
int sgemm_pick_tn(int M, int N, int K, int sms, double* score_out = nullptr) {
  if (score_out != nullptr) *score_out = 1.0;
  if (const int forced = forced_sgemm_tn()) return forced;
  const int nk = ceil_div(K, dgemm::kSgemmBK);
  struct Cfg {
    int tn, per_sm;
    double speed;
  };
  const Cfg cfgs[3] = {{16, 1, 1.00}, {9, 1, 0.93}, {8, 2, 0.92}};
  int best = 16;
  double best_score = -1.0;
  for (const Cfg& c : cfgs) {
    const int bn = dgemm::sgemm_bn(c.tn == 9 ? 8 : c.tn);
    const long long tiles = (long long)ceil_div(M, dgemm::kSgemmBM) * ceil_div(N, bn);
    const long long slots = (long long)c.per_sm * sms;
    double share;
    if (tiles > slots)
      share = 1.0;
    else if (2 * tiles <= slots && nk >= 2)
      share = 2.0 * (double)tiles / (double)slots;
    else
      share = (double)tiles / (double)slots;
    const double score = c.speed * share;
    if (score > best_score + 1e-9) {
      best_score = score;
      best = c.tn;
    }
  }
  if (score_out != nullptr) *score_out = best_score;
  return best;
}

// Below this score of the best whole-K configuration (sgemm_pick_tn), an
// FP32 grid runs as split-K.  Measured on GB300: 1024^3 as two k-halves per
// narrow tile (score 0.81) 55.8 us against 60.4 us as 4 slices; 1000 x 1030
// x 777 (0.91) 59.7 against 67.8 us; 1024 x 2048 x 2048 (0.84, wide) 168
// against 186 us; but 768 x 768 x 4096 (0.45) 101 us as 8 slices against
// 178 us.
constexpr double kSgemmSplitkBelowScore = 0.6;

// Clusters of s CTAs (2, 4, 8) of SGEMM configuration cfg (0 narrow/1,
// 1 narrow/2, 2 wide) that fit at once: the device's answer, else the
// SM count's.
long long sgemm_cluster_cap(const dgemm::SgemmClusterCaps* caps, int sms, int cfg, int s) {
  const int idx = s == 2 ? 0 : (s == 4 ? 1 : 2);
  if (caps != nullptr) return caps->n[cfg][idx];
  return (long long)(cfg == 1 ? 2 : 1) * sms / s;
}

// FP32 plan of the problem as the SGEMM kernel sees it (M x N output, A and
// B with storage ops op_a / op_b, a16 / b16: base and leading dimension
// 16-byte aligned; c_trans: C is stored transposed); the arguments are
// already validated.  caps: the device's cluster capacities (nullptr:
// derived from sms).
gemm_status_t plan_sgemm(int M, int N, int K, int op_a, int op_b, bool a16, bool b16, float beta,
                         int sms, gemm_plan_t* plan, bool c_trans = false,
                         const dgemm::SgemmClusterCaps* caps = nullptr) {
  // TMA cannot transpose 4-byte elements: a transposed operand is staged
  // by the transposing cp.async loaders; with exactly one transposed, the
  // other comes by TMA when it is 16-byte aligned.
  if (!op_a && !op_b)
    plan->path = (a16 && b16) ? GEMM_PATH_SIMT_TMA : GEMM_PATH_SIMT_CPASYNC;
  else if (op_a != op_b && (op_a ? b16 : a16))
    plan->path = GEMM_PATH_SIMT_MIXED;
  else
    plan->path = GEMM_PATH_SIMT_CPASYNC;
  // The two k-halves of a tile can form a cluster (combining in
  // distributed shared memory) only in the row-major kernels.
  const bool row_major = !op_a && !op_b && !c_trans;
  const int narrow_tiles = ceil_div(M, dgemm::kSgemmBM) * ceil_div(N, dgemm::sgemm_bn(8));
  const int nk_all = ceil_div(K, dgemm::kSgemmBK);
  // A grid that no whole-K configuration keeps busy enough runs as split-K
  // (k-slices of narrow tiles into a workspace, then a reduction).  (Eight
  // or four k-slices of a tile as a cluster that adds them in distributed
  // shared memory instead were measured no faster: 256^3 17.0 against
  // 15.0 us, 768^3 31.4 against 31.4 us.)
  double best_score = 1.0;
  sgemm_pick_tn(M, N, K, sms, &best_score);
  int slices = forced_sgemm_tn() || best_score >= kSgemmSplitkBelowScore
                   ? 1
                   : sgemm_splitk_slices(narrow_tiles, sms, nk_all, M, N);
  if (const int fs = forced_sgemm_slices()) {
    const long long slice_bytes = (long long)M * (((long long)N + 3) / 4 * 4) * 4;
    slices = fs < nk_all ? fs : nk_all;
    while (slices > 1 && slices * slice_bytes > kSplitkWorkspaceCap) --slices;
  }
  if (slices > 1) {
    plan->block_m = dgemm::kSgemmBM;
    plan->block_n = dgemm::sgemm_bn(8);
    plan->block_k = dgemm::kSgemmBK;
    plan->stages = dgemm::sgemm_stages(8);
    plan->threads = dgemm::kSgemmThreads;
    plan->tiles = narrow_tiles;
    plan->smem_bytes = dgemm::sgemm_smem_bytes(8);
    plan->split_pieces = 1;
    plan->splitk_slices = slices;
    plan->workspace_bytes = (long long)slices * M * (((long long)N + 3) / 4 * 4) * 4;
    plan->ctas = narrow_tiles * slices;
    return GEMM_OK;
  }
  const int tn = sgemm_pick_tn(M, N, K, sms);
  const int tcfg = tn == 9 ? 8 : tn;   // the tile shape of narrow/1 is narrow's
  plan->block_m = dgemm::kSgemmBM;
  plan->block_n = dgemm::sgemm_bn(tcfg);
  plan->block_k = dgemm::kSgemmBK;
  plan->stages = dgemm::sgemm_stages(tn);
  plan->threads = dgemm::kSgemmThreads;
  plan->tiles = ceil_div(M, dgemm::kSgemmBM) * ceil_div(N, plan->block_n);
  plan->smem_bytes = dgemm::sgemm_smem_bytes(tn);
  // Wave quantisation: with more tiles than resident CTAs the grid is
  // one CTA per slot; all full waves but the last one or two run as whole
  // tiles, and each CTA takes an equal share of the remaining tiles'
  // (tile, k-tile) iteration space (hybrid stream-K); a range boundary
  // inside a tile cuts it into two pieces, which meet through a pair of
  // flag words per boundary.  With beta == 0 the second piece to finish
  // adds into the first one's C; with beta != 0 the first leaves FP32
  // partial sums in a workspace (one tile per boundary) for the second.
  const int slots = (tn == 8 ? 2 : 1) * sms;
  const int nk = ceil_div(K, dgemm::kSgemmBK);
  // A single wave of at most half the slots runs as two CTAs per tile, over
  // the two halves of K: as 2-CTA clusters (two k-slices combining in
  // shared memory) for row-major operands when they all fit at once, else
  // as the stream-K grid of 2 tiles (every boundary in the middle of a
  // tile).
  const int grid = plan->tiles > slots        ? slots
                   : (2 * plan->tiles <= slots && nk >= 2) ? 2 * plan->tiles
                                                           : plan->tiles;
  const int cfg = tn == 9 ? 0 : (tn == 8 ? 1 : 2);
  if (grid == 2 * plan->tiles && row_major && !sgemm_clusters_off() &&
      plan->tiles <= sgemm_cluster_cap(caps, sms, cfg, 2)) {
    plan->split_pieces = 1;
    plan->splitk_slices = 2;
    plan->cluster_ctas = 2;
    plan->ctas = grid;
    return GEMM_OK;
  }
  const int dp_tiles = dgemm::sgemm_dp_tiles(plan->tiles, grid);
  plan->split_tiles = dgemm::sgemm_streamk_cuts(plan->tiles - dp_tiles, nk, grid);
  plan->split_pieces = plan->split_tiles ? 2 : 1;
  plan->splitk_slices = 1;
  if (plan->split_tiles && beta != 0.f)
    plan->workspace_bytes =
        (long long)(grid - 1) * dgemm::kSgemmBM * plan->block_n * 4;
  plan->ctas = grid;
  return GEMM_OK;
}

// pair_clusters: CTA pairs of the pair kernel that can be resident at once
// (0: num_sms / 2, every SM).  allow_copy false: no FP32 operand is copied
// into scratch (transposed or re-pitched) whatever the product's size.
gemm_status_t plan_impl(int dtype, int op_a, int op_b, int M, int N, int K, float alpha,
                        const void* A, int lda, const void* B, int ldb, float beta, const void* C,
                        int ldc, int num_sms, int pair_clusters, gemm_plan_t* plan,
                        bool allow_copy = true,
                        const dgemm::SgemmClusterCaps* caps = nullptr) {
  if (plan == nullptr) return GEMM_ERR_INVALID_ARG;
  std::memset(plan, 0, sizeof(*plan));
  if (dtype < 0 || dtype > 2) return GEMM_ERR_INVALID_ARG;
  if ((op_a != GEMM_OP_N && op_a != GEMM_OP_T) || (op_b != GEMM_OP_N && op_b != GEMM_OP_T))
    return GEMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) {
    plan->path = GEMM_PATH_NOOP;
    return GEMM_OK;
  }
  const int es = dtype == 0 ? 4 : 2;
  if (C == nullptr || ldc < N) return GEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(C) % es) != 0) return GEMM_ERR_INVALID_ARG;
  if (K == 0 || alpha == 0.f) {
    // C := beta * C (zeros when beta == 0); A and B are not read.
    plan->path = GEMM_PATH_ZERO_FILL;
    plan->threads = 256;
    return GEMM_OK;
  }
  if (A == nullptr || B == nullptr) return GEMM_ERR_INVALID_ARG;
  // Stored shapes: A is M x K (op N) or K x M (op T); B is K x N or N x K.
  const int a_rows = op_a ? K : M, a_cols = op_a ? M : K;
  const int b_rows = op_b ? N : K, b_cols = op_b ? K : N;
  if (lda < a_cols || ldb < b_cols) return GEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(A) % es) != 0 || (reinterpret_cast<uintptr_t>(B) % es) != 0)
    return GEMM_ERR_INVALID_ARG;
  const uint64_t cbytes = span_bytes(M, N, ldc, es);
  if (overlap(A, span_bytes(a_rows, a_cols, lda, es), C, cbytes) ||
      overlap(B, span_bytes(b_rows, b_cols, ldb, es), C, cbytes))
    return GEMM_ERR_INVALID_ARG;

  const int sms = num_sms > 0 ? num_sms : 1;
  if (dtype == 0) {
    const bool a16 = aligned16(A) && (lda % 4 == 0), b16 = aligned16(B) && (ldb % 4 == 0);
    // Both operands stored transposed: C^T = B_st . A_st is a product of two
    // row-major arrays, which the kernel computes with TMA staging and
    // stores transposed (SgemmParams::c_trans).
    if (op_a && op_b) return plan_sgemm(N, M, K, 0, 0, b16, a16, beta, sms, plan, true, caps);
    // Exactly one stored transposed: pack it (A into M x K, B into K x N,
    // rows padded to 16 bytes) and run the row-major product, when each
    // packed element is used by at least kPackMinReuse output columns
    // (rows) and the product is large enough to hide the copy's ~6 us of
    // launch and latency.  The copy reads and writes the operand once;
    // staging it transposed with 4-byte cp.async costs the product 13-37 %
    // (measured on GB300: 4096^3 TN +15.6 % staged, +1.3 % packed; 2048^3
    // +32 % / +3.5 %; 1024^3 +16 % / +10 %; 512^3 +17 % / +25 %;
    // 4096 x 128 x 4096 TN +23 % / +30 %).
    if ((op_a || op_b) && allow_copy) {
      const long long rows = op_a ? M : K, cols = op_a ? K : N;
      const long long bytes = rows * ((cols + 3) / 4 * 4) * 4;
      const int reuse = op_a ? N : M;
      const int forced = forced_sgemm_pack();
      const bool pack = forced == 1 || (forced == -1 && reuse >= kPackMinReuse &&
                                        (long long)M * N * K >= kPackMinWork &&
                                        bytes <= kPackCapBytes);
      if (pack) {
        // The other (row-major) operand is re-pitched as well when TMA
        // cannot address it (the product is far above kRepitchMinWork) and
        // both copies fit under the cap.
        const bool other16 = op_a ? b16 : a16;
        const long long other =
            (op_a ? (long long)K * round4(N) : (long long)M * round4(K)) * 4;
        const long long total = (bytes + 255) / 256 * 256 + (other + 255) / 256 * 256;
        const bool both = !other16 && total <= kPackCapBytes;
        const gemm_status_t st =
            plan_sgemm(M, N, K, 0, 0, true, both || other16, beta, sms, plan, false, caps);
        plan->pack = (op_a ? 1 : 2) | (both ? (op_a ? 2 : 1) : 0);
        plan->pack_bytes = both ? total : bytes;
        return st;
      }
    }
    // Row-major operands whose base or leading dimension is not 16-byte
    // aligned cannot be staged by TMA; 4-byte cp.async staging costs the
    // product ~35 % (FMA pipe 57 % busy against 82 %).  Large enough
    // products first copy such an operand into scratch with 16-byte rows
    // (HBM-bound, every element read and written once) and run with TMA.
    if (!op_a && !op_b && (!a16 || !b16) && allow_copy) {
      const long long bytes_a = a16 ? 0 : (long long)M * round4(K) * 4;
      const long long bytes_b = b16 ? 0 : (long long)K * round4(N) * 4;
      const long long bytes = (bytes_a + 255) / 256 * 256 + bytes_b;
      const int forced = forced_sgemm_repitch();
      if (forced == 1 || (forced == -1 && (long long)M * N * K >= kRepitchMinWork &&
                          bytes <= kPackCapBytes)) {
        const gemm_status_t st =
            plan_sgemm(M, N, K, 0, 0, true, true, beta, sms, plan, false, caps);
        plan->pack = (a16 ? 0 : 1) | (b16 ? 0 : 2);
        plan->pack_bytes = bytes;
        return st;
      }
    }
    return plan_sgemm(M, N, K, op_a, op_b, a16, b16, beta, sms, plan, false, caps);
  }
  // FP16 / BF16: TMA in and out needs 16-byte aligned bases and pitches.
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || (lda % 8) || (ldb % 8) || (ldc % 8))
    return GEMM_ERR_MISALIGNED;
  plan->path = GEMM_PATH_TC_TMA;
  plan->threads = dgemm::kTcThreads;
  plan->cluster_ctas = 1;
  // CTA pairs (256 x 256 tiles, half of B staged per SM, 128-deep stages)
  // unless single CTAs keep clearly more SMs busy in their first round
  // (column parts or split-K on a small grid): with the same SMs busy the
  // pair kernel was measured 1.06-1.17x faster (2048^3: 21.2 vs 22.6 us;
  // 2048 x 2048 x 8192: 54.3 vs 63.5 us), so it wins unless
  // 1.15 x its busy SMs < the single kernel's.
  // The pair grid is persistent: at most as many pairs as fit at once.  A
  // hand-over of FP32 partials between pairs (the K split) polls for a
  // partial that another pair computes, so it needs every pair of the grid
  // resident together; when fewer clusters than sms / 2 fit (a GPU shared
  // with other work, or partitioned), it is not used.
  const int all_pairs = sms / 2;
  const int pairs = pair_clusters > 0 && pair_clusters < all_pairs ? pair_clusters : all_pairs;
  const bool handover = pair_clusters <= 0 || pair_clusters >= all_pairs;
  const int pair_tiles = ceil_div(M, 2 * dgemm::kTc2BM) * ceil_div(N, dgemm::kTc2BN);
  const int forced = forced_tc_kernel();
  const auto single_busy = [&]() {
    const int tiles1 = ceil_div(M, dgemm::kTcBM) * ceil_div(N, dgemm::kTcBN);
    const dgemm::TcSplit parts = dgemm::tc_split(tiles1, sms);
    const bool fill = parts.split_tiles == tiles1 && 4 * parts.parts * tiles1 >= 3 * sms;
    const int slices =
        fill ? 1 : splitk_slices_capped(tiles1, sms, ceil_div(K, dgemm::kTcBK), M, N);
    const long long units = slices > 1 ? (long long)tiles1 * slices
                                       : tiles1 + (long long)parts.split_tiles * (parts.parts - 1);
    return units < sms ? (int)units : sms;
  };
  const int nk_pair = ceil_div(K, dgemm::kTc2BK);
  // The pair kernel's tiles beyond whole rounds: a stream-K share of the
  // last two rounds when K is long enough, else the last round's tiles as
  // column parts when they fit it twice.
  const int sk_first = (tc_streamk_disabled() || !handover)
                           ? -1
                           : dgemm::tc_pair_streamk_first(pair_tiles, pairs, nk_pair,
                                                          tc_sk_min_rounds());
  const auto pair_busy = [&]() {
    if (sk_first >= 0) return 2 * pairs;
    const dgemm::TcSplit sp = dgemm::tc_pair_split(pair_tiles, pairs);
    const int units = pair_tiles + sp.split_tiles * (sp.parts - 1);
    return 2 * (units < pairs ? units : pairs);
  };
  const bool use_pairs =
      forced == 2 || (forced == 0 && 115LL * pair_busy() >= 100LL * single_busy());
  if (pairs >= 1 && use_pairs) {
    plan->cluster_ctas = 2;
    plan->block_m = 2 * dgemm::kTc2BM;
    plan->block_n = dgemm::kTc2BN;
    plan->block_k = dgemm::kTc2BK;
    plan->stages = dgemm::kTc2Stages;
    plan->tiles = pair_tiles;
    plan->splitk_slices = 1;
    if (sk_first >= 0) {
      // Cut tiles: a head on one pair, a tail on the next; one 256 x 256
      // FP32 head partial per range boundary in the workspace.
      plan->split_tiles = dgemm::tc_pair_streamk_cuts(pair_tiles - sk_first, pairs, nk_pair);
      plan->split_pieces = plan->split_tiles ? 2 : 1;
      plan->split_in_k = 1;
      plan->streamk_first_tile = sk_first;
      plan->workspace_bytes = (long long)pairs * 2 * dgemm::kTc2BM * dgemm::kTc2BN * 4;
      plan->ctas = 2 * pairs;
    } else {
      dgemm::TcSplit sp = dgemm::tc_pair_split(pair_tiles, pairs);
      if (tc_split_disabled()) sp = dgemm::TcSplit{0, 1};
      plan->split_tiles = sp.split_tiles;
      plan->split_pieces = sp.parts;
      plan->streamk_first_tile = -1;
      const int units = pair_tiles + sp.split_tiles * (sp.parts - 1);
      plan->ctas = 2 * (units < pairs ? units : pairs);
    }
    plan->smem_bytes = dgemm::kTc2SmemBytes;
    return GEMM_OK;
  }
  plan->block_m = dgemm::kTcBM;
  plan->block_n = dgemm::kTcBN;
  plan->block_k = dgemm::kTcBK;
  plan->stages = dgemm::kTcStages;
  plan->tiles = ceil_div(M, dgemm::kTcBM) * ceil_div(N, dgemm::kTcBN);
  plan->smem_bytes = dgemm::kTcSmemBytes;
  // A grid filling at most half of the SMs with a long K runs as split-K,
  // unless splitting every tile into column parts (full K each) already
  // fills three quarters of the SMs: that needs no workspace and no second
  // launch (1024^3 FP16: 22.5 us with split-K; a launch alone costs ~4.5 us).
  const dgemm::TcSplit parts_only = dgemm::tc_split(plan->tiles, sms);
  const bool parts_fill = parts_only.split_tiles == plan->tiles &&
                          4 * parts_only.parts * plan->tiles >= 3 * sms;
  const int slices = (tc_split_disabled() || parts_fill)
                         ? 1
                         : splitk_slices_capped(plan->tiles, sms, ceil_div(K, dgemm::kTcBK), M, N);
  if (slices > 1) {
    plan->split_pieces = 1;
    plan->splitk_slices = slices;
    plan->workspace_bytes = (long long)slices * M * (((long long)N + 3) / 4 * 4) * 4;
    const int units = plan->tiles * slices;
    plan->ctas = units < sms ? units : sms;
    return GEMM_OK;
  }
  dgemm::TcSplit sp = dgemm::tc_split(plan->tiles, sms);
  if (tc_split_disabled()) sp = dgemm::TcSplit{0, 1};
  plan->split_tiles = sp.split_tiles;
  plan->split_pieces = sp.parts;
  plan->splitk_slices = 1;
  const int units = plan->tiles + sp.split_tiles * (sp.parts - 1);
  plan->ctas = units < sms ? units : sms;
  plan->smem_bytes = dgemm::kTcSmemBytes;
  return GEMM_OK;
}

// The tile-schedule fields of TcParams for an FP16/BF16 plan (single CTAs
// or pairs); the kernels and gemm_pair_units read them the same way.
void tc_schedule_params(const gemm_plan_t& plan, int M, int N, dgemm::TcParams* p) {
  p->tiles_m = ceil_div(M, plan.block_m);
  p->tiles_n = ceil_div(N, plan.block_n);
  p->group_m = tc_group_override() > 0    ? tc_group_override()
               : plan.cluster_ctas == 2 ? dgemm::kTc2GroupM
                                        : dgemm::kTcGroupM;
  p->full_tiles = plan.tiles - plan.split_tiles;
  p->split_tiles = plan.split_tiles;
  p->parts = plan.split_pieces;
  p->slices = plan.splitk_slices;
  p->sk = 0;
  if (plan.cluster_ctas == 2 && plan.split_in_k) {
    p->sk = 1;
    p->sk_first_tile = plan.streamk_first_tile;
    p->sk_tiles = plan.tiles - plan.streamk_first_tile;
    p->full_tiles = plan.tiles;
    p->split_tiles = 0;
    p->parts = 1;
  }
}

// fixed: flag words and split-K workspace supplied by the caller
// (gemm_f32_noalloc) instead of the stream's library-owned arrays.
gemm_status_t run(int dtype, int op_a, int op_b, int M, int N, int K, float alpha, const void* A,
                  int lda, const void* B, int ldb, float beta, void* C, int ldc,
                  cudaStream_t stream, bool allow_copy = true,
                  const dgemm::FixedScratch* fixed = nullptr) {
  gemm_plan_t plan;
  gemm_status_t st = plan_impl(dtype, op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                               1, 0, &plan, allow_copy);
  if (st != GEMM_OK) return st;
  if (plan.path == GEMM_PATH_NOOP) return GEMM_OK;
  DeviceInfo* dev = nullptr;
  st = current_device(&dev);
  if (st != GEMM_OK) return st;
  // Re-plan with the device's SM count (validation above needs no device).
  st = plan_impl(dtype, op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dev->sms,
                 dev->pair_clusters, &plan, allow_copy, &dev->sgemm_caps);
  if (st != GEMM_OK) return st;
  cudaError_t e = cudaSuccess;

  if (plan.path == GEMM_PATH_ZERO_FILL) {
    e = dgemm::launch_scale_c(C, M, N, ldc, dtype, beta, stream);
  } else if (dtype == 0) {
    // The kernel's view: with both operands stored transposed it computes
    // C^T = B_st . A_st (N x M, row-major operands) and stores C transposed.
    const bool swap = op_a && op_b;
    const int kM = swap ? N : M, kN = swap ? M : N;
    const void* kA = swap ? B : A;
    const void* kB = swap ? A : B;
    int klda = swap ? ldb : lda, kldb = swap ? lda : ldb;
    int kop_a = swap ? 0 : op_a, kop_b = swap ? 0 : op_b;
    if (plan.pack) {
      // Each copied operand becomes row-major with 16-byte rows in scratch:
      // A stored K x M is transposed into M x K, B stored N x K into K x N;
      // row-major operands are re-pitched, both in one launch.  A's copy
      // comes first.
      float* packed = nullptr;
      st = get_workspace(stream, (size_t)plan.pack_bytes, &packed, kWsPack);
      if (st != GEMM_OK) return st;
      float* dst = packed;
      dgemm::RepitchJob jobs[2];
      int njobs = 0;
      for (int which = 0; which < 2 && e == cudaSuccess; ++which) {
        if (!(plan.pack & (1 << which))) continue;
        const bool is_a = which == 0;
        const bool trans = is_a ? op_a != 0 : op_b != 0;
        const long long rows = is_a ? M : K, cols = is_a ? K : N;   // of the copy
        const long long ldp = round4(cols);
        const float* src = static_cast<const float*>(is_a ? A : B);
        const long long lds = is_a ? lda : ldb;
        if (trans)
          e = dgemm::launch_transpose_f32(src, cols, rows, lds, dst, ldp, dev->sms, stream);
        else
          jobs[njobs++] = dgemm::RepitchJob{src, rows, cols, lds, dst, ldp};
        if (is_a) {
          kA = dst;
          klda = (int)ldp;
          kop_a = 0;
        } else {
          kB = dst;
          kldb = (int)ldp;
          kop_b = 0;
        }
        dst += (rows * ldp + 63) / 64 * 64;
      }
      if (e == cudaSuccess && njobs > 0)
        e = dgemm::launch_repitch_f32(jobs, njobs, dev->sms, stream);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
      }
    }
    dgemm::SgemmParams p;
    p.M = kM;
    p.N = kN;
    p.K = K;
    p.op_a = kop_a;
    p.op_b = kop_b;
    p.c_trans = swap ? 1 : 0;
    p.A = static_cast<const float*>(kA);
    p.lda = klda;
    p.B = static_cast<const float*>(kB);
    p.ldb = kldb;
    p.C = static_cast<float*>(C);
    p.ldc = ldc;
    // CTA pairs over K (a plan of 2 k-slices in 2-CTA clusters) run the
    // stream-K schedule of a grid of 2 tiles (each CTA one half of a tile)
    // with the cluster exchange, on the plan's tile configuration.
    const bool cluster = plan.cluster_ctas > 1;
    const int tn = plan.splitk_slices > 1 && !cluster ? 8 : sgemm_pick_tn(kM, kN, K, dev->sms);
    p.tiles_m = ceil_div(kM, dgemm::kSgemmBM);
    p.tiles_n = ceil_div(kN, plan.block_n);
    p.grid = plan.ctas;
    p.dp_tiles = plan.splitk_slices > 1 ? 0 : dgemm::sgemm_dp_tiles(plan.tiles, plan.ctas);
    p.split_tiles = plan.split_tiles;
    p.slices = cluster ? 1 : plan.splitk_slices;
    p.cluster_k = cluster ? 1 : 0;
    p.ws = nullptr;
    p.ldw = ((long long)kN + 3) / 4 * 4;
    if (p.slices > 1) {
      if (fixed != nullptr) {
        if (plan.workspace_bytes > fixed->ws_bytes) return GEMM_ERR_SCRATCH_LIMIT;
        p.ws = fixed->ws;
      } else {
        st = get_workspace(stream, (size_t)plan.workspace_bytes, &p.ws);
        if (st != GEMM_OK) return st;
      }
    }
    if (p.slices == 1 && plan.split_tiles > 0) {
      if (plan.workspace_bytes > 0) {
        if (fixed != nullptr) return GEMM_ERR_SCRATCH_LIMIT;   // (beta != 0: never planned)
        st = get_workspace(stream, (size_t)plan.workspace_bytes, &p.tail_ws);
        if (st != GEMM_OK) return st;
      }
      const long long words = 2ll * (plan.ctas - 1);
      if (fixed != nullptr) {
        if (words > fixed->flag_words) return GEMM_ERR_SCRATCH_LIMIT;
        p.sk_flags = fixed->flags;
        p.epoch = fixed->epoch;
      } else {
        float* flags = nullptr;
        st = get_workspace(stream, (size_t)words * 4, &flags, kWsFlags);
        if (st != GEMM_OK) return st;
        p.sk_flags = reinterpret_cast<unsigned*>(flags);
        p.epoch = next_epoch(stream);
      }
    }
    p.alpha = alpha;
    p.beta = beta;
    p.c_vec4 = aligned16(C) && (ldc % 4 == 0) && (swap || N % 4 == 0);
    p.fault = dev->fault;
    p.timeout_ns = wait_timeout_ns();
    const bool tma = plan.path == GEMM_PATH_SIMT_TMA || plan.path == GEMM_PATH_SIMT_MIXED;
    alignas(64) CUtensorMap tmA{}, tmB{};
    // (Mixed staging: only the operand that is not transposed has a map.)
    if (tma && !kop_a &&
        !encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, kA, (uint64_t)K, (uint64_t)kM,
                   (uint64_t)klda * 4, dgemm::kSgemmBK, dgemm::kSgemmBM,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return GEMM_ERR_LAUNCH;
    if (tma && !kop_b &&
        !encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, kB, (uint64_t)kN, (uint64_t)K,
                   (uint64_t)kldb * 4, (uint32_t)plan.block_n, dgemm::kSgemmBK,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
      return GEMM_ERR_LAUNCH;
    e = dgemm::launch_sgemm(p, tn, tma, &tmA, &tmB, stream);
    if (e == cudaSuccess && p.slices > 1)
      e = dgemm::launch_splitk_reduce(p.ws, p.slices, kM, kN, p.ldw, C, ldc, 0, alpha, beta,
                                      stream, p.c_trans);
  } else {
    const CUtensorMapDataType dt =
        dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    alignas(64) CUtensorMap tmA, tmB, tmC;
    // A: {K, M} with 64 x 128 boxes, or as stored K x M ({M, K}, 64 x 64
    // boxes); B: {N, K} with 64 x 64 boxes (64 x 128 for CTA pairs: one box
    // per 64-column block and stage), or as stored N x K ({K, N}).
    const bool enc_a =
        op_a ? encode_2d(&tmA, dt, A, (uint64_t)M, (uint64_t)K, (uint64_t)lda * 2, 64,
                         dgemm::kTcBK, CU_TENSOR_MAP_SWIZZLE_128B)
             : encode_2d(&tmA, dt, A, (uint64_t)K, (uint64_t)M, (uint64_t)lda * 2, dgemm::kTcBK,
                         dgemm::kTcBM, CU_TENSOR_MAP_SWIZZLE_128B);
    const bool enc_b =
        op_b ? encode_2d(&tmB, dt, B, (uint64_t)K, (uint64_t)N, (uint64_t)ldb * 2, dgemm::kTcBK,
                         64, CU_TENSOR_MAP_SWIZZLE_128B)
             : encode_2d(&tmB, dt, B, (uint64_t)N, (uint64_t)K, (uint64_t)ldb * 2, 64,
                         plan.cluster_ctas == 2 ? dgemm::kTc2BK : dgemm::kTcBK,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    // C up to the last whole 16-byte granule of a row; the kernels write the
    // ragged tail (N % 8 columns) with plain stores.
    const int n_tma = N & ~7;
    if (!enc_a || !enc_b ||
        !encode_2d(&tmC, dt, C, (uint64_t)(n_tma > 0 ? n_tma : N), (uint64_t)M,
                   (uint64_t)ldc * 2, dgemm::kTcEpiCols, 32, CU_TENSOR_MAP_SWIZZLE_128B))
      return GEMM_ERR_LAUNCH;
    dgemm::TcParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.op_a = op_a;
    p.op_b = op_b;
    tc_schedule_params(plan, M, N, &p);
    p.ws = nullptr;
    p.ldw = ((long long)N + 3) / 4 * 4;
    if (p.slices > 1) {
      st = get_workspace(stream, (size_t)plan.workspace_bytes, &p.ws);
      if (st != GEMM_OK) return st;
    }
    p.alpha = alpha;
    p.beta = beta;
    p.c_in = C;
    p.c_out = C;
    p.ldc = ldc;
    p.n_tma = n_tma;
    p.fault = dev->fault;
    p.timeout_ns = wait_timeout_ns();
    if (plan.cluster_ctas == 2 && plan.split_in_k) {
      // Stream-K share: head partials and their flags, one per range
      // boundary (boundary 0 is unused).
      st = get_workspace(stream, (size_t)plan.workspace_bytes, &p.kpart);
      if (st != GEMM_OK) return st;
      float* flags = nullptr;
      st = get_workspace(stream, (size_t)(plan.ctas / 2) * 8 * 4, &flags, kWsFlags);
      if (st != GEMM_OK) return st;
      p.kflag = reinterpret_cast<unsigned*>(flags);
      p.epoch = next_epoch(stream);
    }
    if (plan.cluster_ctas == 2)
      e = dgemm::launch_gemm_tc_pair(dtype, p, &tmA, &tmB, &tmC, plan.ctas / 2, stream);
    else
      e = dgemm::launch_gemm_tc(dtype, p, &tmA, &tmB, &tmC, plan.ctas, stream);
    if (e == cudaSuccess && p.slices > 1)
      e = dgemm::launch_splitk_reduce(p.ws, p.slices, M, N, p.ldw, C, ldc, dtype, alpha, beta,
                                      stream);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

}  // namespace

namespace dgemm {

// For other translation units of the library: the current device's fault
// word (nullptr if the device is unsupported) and the bound of every wait.
unsigned* current_fault_word() {
  DeviceInfo* dev = nullptr;
  return current_device(&dev) == GEMM_OK ? dev->fault : nullptr;
}
unsigned long long wait_bound_ns() { return wait_timeout_ns(); }

gemm_status_t run_f32_no_copy(int M, int N, int K, const float* A, int lda, const float* B,
                              int ldb, float* C, int ldc, cudaStream_t stream,
                              const FixedScratch& scratch) {
  return run(0, GEMM_OP_N, GEMM_OP_N, M, N, K, 1.f, A, lda, B, ldb, 0.f, C, ldc, stream, false,
             &scratch);
}

bool pdl_enabled() {
  static const bool v = [] {
    const char* s = std::getenv("DENSE_GEMM_PDL");
    return !(s != nullptr && std::strcmp(s, "0") == 0);
  }();
  return v;
}

}  // namespace dgemm

extern "C" {

gemm_status_t gemm_f32(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                       float* C, int ldc, cudaStream_t stream) {
  return run(0, GEMM_OP_N, GEMM_OP_N, M, N, K, 1.f, A, lda, B, ldb, 0.f, C, ldc, stream);
}

gemm_status_t gemm_f16(int M, int N, int K, const gemm_half_t* A, int lda, const gemm_half_t* B,
                       int ldb, gemm_half_t* C, int ldc, cudaStream_t stream) {
  return run(1, GEMM_OP_N, GEMM_OP_N, M, N, K, 1.f, A, lda, B, ldb, 0.f, C, ldc, stream);
}

gemm_status_t gemm_bf16(int M, int N, int K, const gemm_bfloat16_t* A, int lda,
                        const gemm_bfloat16_t* B, int ldb, gemm_bfloat16_t* C, int ldc,
                        cudaStream_t stream) {
  return run(2, GEMM_OP_N, GEMM_OP_N, M, N, K, 1.f, A, lda, B, ldb, 0.f, C, ldc, stream);
}

gemm_status_t gemm_f32_ex(int M, int N, int K, float alpha, const float* A, int lda,
                          const float* B, int ldb, float beta, float* C, int ldc,
                          cudaStream_t stream) {
  return run(0, GEMM_OP_N, GEMM_OP_N, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

gemm_status_t gemm_f16_ex(int M, int N, int K, float alpha, const gemm_half_t* A, int lda,
                          const gemm_half_t* B, int ldb, float beta, gemm_half_t* C, int ldc,
                          cudaStream_t stream) {
  return run(1, GEMM_OP_N, GEMM_OP_N, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

gemm_status_t gemm_bf16_ex(int M, int N, int K, float alpha, const gemm_bfloat16_t* A, int lda,
                           const gemm_bfloat16_t* B, int ldb, float beta, gemm_bfloat16_t* C,
                           int ldc, cudaStream_t stream) {
  return run(2, GEMM_OP_N, GEMM_OP_N, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

gemm_status_t gemm_f32_op(gemm_op_t op_a, gemm_op_t op_b, int M, int N, int K, float alpha,
                          const float* A, int lda, const float* B, int ldb, float beta, float* C,
                          int ldc, cudaStream_t stream) {
  return run(0, op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

gemm_status_t gemm_f16_op(gemm_op_t op_a, gemm_op_t op_b, int M, int N, int K, float alpha,
                          const gemm_half_t* A, int lda, const gemm_half_t* B, int ldb, float beta,
                          gemm_half_t* C, int ldc, cudaStream_t stream) {
  return run(1, op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

gemm_status_t gemm_bf16_op(gemm_op_t op_a, gemm_op_t op_b, int M, int N, int K, float alpha,
                           const gemm_bfloat16_t* A, int lda, const gemm_bfloat16_t* B, int ldb,
                           float beta, gemm_bfloat16_t* C, int ldc, cudaStream_t stream) {
  return run(2, op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

const char* gemm_status_string(gemm_status_t status) {
  switch (status) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_INVALID_ARG: return "invalid argument (size, leading dimension, null or overlap)";
    case GEMM_ERR_MISALIGNED: return "operand base or leading dimension not 16-byte aligned";
    case GEMM_ERR_UNSUPPORTED_DEVICE: return "no current CUDA device of compute capability 10.3";
    case GEMM_ERR_LAUNCH: return "kernel launch failed";
    case GEMM_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait gave up";
    case GEMM_ERR_SCRATCH_LIMIT:
      return "split-K problem needs more scratch than the 16 MiB static array of gemm_f32_noalloc";
  }
  return "unknown status";
}

gemm_status_t gemm_device_check(cudaStream_t stream, unsigned* fault_bits) {
  if (fault_bits) *fault_bits = 0;
  DeviceInfo* dev = nullptr;
  gemm_status_t st = current_device(&dev);
  if (st != GEMM_OK) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  unsigned v = 0;
  if (cudaMemcpy(&v, dev->fault, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  if (fault_bits) *fault_bits = v;
  if (v != 0) {
    const unsigned zero = 0;
    cudaMemcpy(dev->fault, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    return GEMM_ERR_DEVICE_TIMEOUT;
  }
  return GEMM_OK;
}

gemm_status_t gemm_plan(int dtype, int M, int N, int K, const void* A, int lda, const void* B,
                        int ldb, const void* C, int ldc, int num_sms, gemm_plan_t* plan) {
  return plan_impl(dtype, GEMM_OP_N, GEMM_OP_N, M, N, K, 1.f, A, lda, B, ldb, 0.f, C, ldc,
                   num_sms, 0, plan);
}

gemm_status_t gemm_plan_ex(int dtype, int M, int N, int K, float alpha, const void* A, int lda,
                           const void* B, int ldb, float beta, const void* C, int ldc,
                           int num_sms, gemm_plan_t* plan) {
  return plan_impl(dtype, GEMM_OP_N, GEMM_OP_N, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                   num_sms, 0, plan);
}

gemm_status_t gemm_plan_op(int dtype, gemm_op_t op_a, gemm_op_t op_b, int M, int N, int K,
                           float alpha, const void* A, int lda, const void* B, int ldb,
                           float beta, const void* C, int ldc, int num_sms, gemm_plan_t* plan) {
  return plan_impl(dtype, op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, num_sms, 0,
                   plan);
}

gemm_status_t gemm_plan_resident(int dtype, gemm_op_t op_a, gemm_op_t op_b, int M, int N, int K,
                                 float alpha, const void* A, int lda, const void* B, int ldb,
                                 float beta, const void* C, int ldc, int num_sms,
                                 int pair_clusters, gemm_plan_t* plan) {
  if (pair_clusters < 0) return GEMM_ERR_INVALID_ARG;
  return plan_impl(dtype, op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, num_sms,
                   pair_clusters, plan);
}

int gemm_pair_units(const gemm_plan_t* plan, int M, int N, int K, int pair, int* units,
                    int max_units) {
  if (plan == nullptr || plan->path != GEMM_PATH_TC_TMA || plan->cluster_ctas != 2 || M <= 0 ||
      N <= 0 || K <= 0 || pair < 0 || pair >= plan->ctas / 2 || max_units < 0 ||
      (max_units > 0 && units == nullptr))
    return -1;
  dgemm::TcParams p;
  tc_schedule_params(*plan, M, N, &p);
  const int nk = ceil_div(K, dgemm::kTc2BK);
  const dgemm::TcPairSched s = dgemm::tc_pair_sched(pair, plan->ctas / 2, p, nk);
  for (int j = 0; j < s.n && j < max_units; ++j) {
    const dgemm::TcUnit w = dgemm::tc_pair_unit(s, j, plan->ctas / 2, p, nk);
    const int v[8] = {w.tm, w.tn, w.n_off, w.n_w, w.kb, w.ke, w.kind, w.slot};
    for (int i = 0; i < 8; ++i) units[8 * j + i] = v[i];
  }
  return s.n;
}

int gemm_pair_clusters(void) {
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != GEMM_OK) return -1;
  return dev->pair_clusters;
}

int gemm_sgemm_clusters(int config, int cluster_size) {
  if (config < 0 || config > 2 || (cluster_size != 2 && cluster_size != 4 && cluster_size != 8))
    return -1;
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != GEMM_OK) return -1;
  return dev->sgemm_caps.n[config][cluster_size == 2 ? 0 : (cluster_size == 4 ? 1 : 2)];
}

int gemm_smem_layout_offset(int layout, int row, int col) {
  if (layout == 0) {
    if (row < 0 || row >= dgemm::kSgemmBM || col < 0 || col >= dgemm::kSgemmBK) return -1;
    return dgemm::sgemm_smem_offset(0, 0, row, col);
  }
  if (layout >= 1 && layout <= 4) {
    const int bn = dgemm::sgemm_bn(layout == 1 || layout == 3 ? 8 : 16);
    if (row < 0 || row >= dgemm::kSgemmBK || col < 0 || col >= bn) return -1;
    return dgemm::sgemm_smem_offset(layout <= 2 ? 1 : 2, bn, row, col);
  }
  return -1;
}

gemm_status_t gemm_selftest_timeout(unsigned timeout_us, cudaStream_t stream) {
  DeviceInfo* dev = nullptr;
  gemm_status_t st = current_device(&dev);
  if (st != GEMM_OK) return st;
  if (dgemm::launch_selftest_timeout(dev->fault, (unsigned long long)timeout_us * 1000ull,
                                     stream) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

gemm_status_t gemm_selftest_flag_timeout(unsigned timeout_us, cudaStream_t stream) {
  DeviceInfo* dev = nullptr;
  gemm_status_t st = current_device(&dev);
  if (st != GEMM_OK) return st;
  if (dgemm::launch_selftest_flag_timeout(dev->fault, (unsigned long long)timeout_us * 1000ull,
                                          stream) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

}  // extern "C"
