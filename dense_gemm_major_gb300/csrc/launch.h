// Internal interface between the C-ABI dispatcher (api.cu) and the kernel
// translation units.  Not installed; callers use include/dense_gemm.h.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

namespace dgemm {

// ---------------------------------------------------------------- FP32 SIMT

// Two tile configurations, both 256 threads (8 warps as 4 x 2, each warp a
// 4 x 8 lane grid), BM = 128, BK = 32, TM = 8 rows per thread:
//   narrow: TN = 8  -> 8 x 8 per thread,  BN = 128, 3 stages, 2 CTAs per SM;
//   wide:   TN = 16 -> 8 x 16 per thread, BN = 256, 4 stages, 1 CTA per SM.
constexpr int kSgemmBM = 128;
constexpr int kSgemmBK = 32;
constexpr int kSgemmThreads = 256;
constexpr int kSgemmGroupM = 16;   // tile rows per rasterisation group (L2 reuse)
constexpr int sgemm_bn(int tn) { return 16 * tn; }
constexpr int sgemm_stages(int tn) { return tn == 8 ? 3 : 4; }
constexpr int sgemm_smem_bytes(int tn) {
  return sgemm_stages(tn) * (kSgemmBM * kSgemmBK + kSgemmBK * sgemm_bn(tn)) * 4 + 1024 /*align*/ +
         64 /*barriers*/;
}

struct SgemmParams {
  int M, N, K;
  // op_a = 1: A stored K x M, element (i,k) at A[k*lda + i]; op_b = 1: B
  // stored N x K, element (k,j) at B[j*ldb + k] (cp.async staging only).
  int op_a = 0, op_b = 0;
  const float* A;
  long long lda;
  const float* B;
  long long ldb;
  float* C;
  long long ldc;
  int tiles_m, tiles_n;
  // Hybrid stream-K schedule (slices == 1), grid G: CTA c computes the
  // whole tiles c, c + G, ... below dp_tiles, then the k-tiles
  // [c * total / G, (c + 1) * total / G) of the iteration space of the
  // remaining tiles, total = (tiles - dp_tiles) * nk (G <= tiles - dp_tiles,
  // or G = 2 tiles with dp_tiles = 0), one unit per tile it touches.
  // split_tiles tiles are cut by a range boundary into two pieces.  With
  // tail_ws == nullptr (only when beta = 0) both pieces add alpha times
  // their FP32 partial sums into C, which is zeroed first; with exactly two
  // addends the result does not depend on their order.  Otherwise the
  // pieces of the tile cut by boundary c store their partial sums at
  // tail_ws + (2 (c - 1) + piece) * BM * BN (row-major, leading dimension
  // BN) and a fixup kernel writes alpha * (piece 0 + piece 1) + beta * C, in
  // that order, so the result is again independent of scheduling.
  int grid;
  int dp_tiles = 0;
  int split_tiles;
  float* tail_ws = nullptr;
  // Split-K mode (slices > 1): CTA u computes k-slice u % slices of tile
  // u / slices (k-tiles [s*nk/slices, (s+1)*nk/slices)) and stores its FP32
  // partial tile at ws + s * M * ldw (row-major, leading dimension ldw);
  // splitk_reduce then sums the slices in slice order into C.  grid and
  // split_tiles are unused in this mode.
  int slices;
  float* ws;
  long long ldw;
  // C := alpha * (A.B) + beta * C; the old C is read only when beta != 0
  // (in split-K mode splitk_reduce applies alpha and beta; for split tiles
  // with tail_ws the fixup kernel does).
  float alpha = 1.f, beta = 0.f;
  int c_vec4;        // C rows may be written with 16-byte stores (C and ldc
                     // 16-byte aligned; row-major C also needs N % 4 == 0,
                     // a transposed C checks each 4-row block against M)
  // c_trans = 1: the kernel's output element (r, c) lives at C[c * ldc + r]
  // (the product is computed as C^T = B_st . A_st for operands both stored
  // transposed); C is then read and written element by element.
  int c_trans = 0;
  unsigned* fault;   // device fault word
  unsigned long long timeout_ns;
};

// Tile (tm, tn) of linear tile index t under grouped rasterisation: tiles
// walk down a group of `group` tile rows before moving one tile column right.
__host__ __device__ inline void grouped_tile(int t, int tiles_m, int tiles_n, int group, int& tm,
                                             int& tn) {
  const int per_group = group * tiles_n;
  const int g = t / per_group;
  const int first_m = g * group;
  const int gsize = (tiles_m - first_m) < group ? (tiles_m - first_m) : group;
  const int r = t - g * per_group;
  tm = first_m + r % gsize;
  tn = r / gsize;
}

// tn: 8 (narrow) or 16 (wide).  use_tma: A and B are staged by TMA
// (16-byte aligned bases and strides); otherwise by 4-byte cp.async with
// zero fill.  When p.split_tiles > 0, first zeroes C on the cut tiles
// (tail_ws == nullptr) or afterwards combines their pieces (one extra launch
// either way).  Returns the launch error.
cudaError_t launch_sgemm(const SgemmParams& p, int tn, bool use_tma, const CUtensorMap* tmA,
                         const CUtensorMap* tmB, cudaStream_t stream);

// The kernels for p.op_a or p.op_b set: the transposed operand(s) staged
// by transposing cp.async copies; with use_tma (exactly one operand
// transposed, the other 16-byte aligned) the other operand by TMA through
// its tensor map.  tn 16 or 8 (9 is run as 8), launched like launch_sgemm.
cudaError_t launch_sgemm_op(const SgemmParams& p, int tn, bool use_tma, const CUtensorMap* tmA,
                            const CUtensorMap* tmB, cudaStream_t stream);

// Element offset of (row, col) inside one stage of the FP32 A tile
// (which = 0), the B tile of a BN-wide configuration (which = 1) or the B
// tile of a transposed B (which = 2); host copy of the device layout.
int sgemm_smem_offset(int which, int bn, int r, int c);

// Whole tiles a hybrid stream-K schedule of `tiles` tiles on `grid` CTAs
// computes in full waves before sharing out the rest: all waves but the
// last one or two, so that at least `grid` tiles are left.
inline int sgemm_dp_tiles(int tiles, int grid) {
  return tiles / grid >= 2 ? (tiles / grid - 1) * grid : 0;
}

// Stream-K share of `tiles` tiles of nk k-tiles each on `grid` CTAs (grid <=
// tiles, or grid = 2 tiles): returns the number of tiles a range boundary
// c * tiles * nk / grid cuts (the kernel's rule).
inline int sgemm_streamk_cuts(int tiles, int nk, int grid) {
  if (grid <= 1 || nk <= 0) return 0;
  const long long total = (long long)tiles * nk;
  int cuts = 0;
  for (int c = 1; c < grid; ++c)
    if (((long long)c * total / grid) % nk != 0) ++cuts;
  return cuts;
}

// ---------------------------------------------------------------- FP16/BF16 tcgen05

// Output tile 128 x 256 per CTA (one tcgen05.mma M=128, N=256 accumulator,
// double-buffered in tensor memory), k-tile 64, 4-stage TMA ring, persistent
// grid of at most one CTA per SM.
constexpr int kTcBM = 128;
constexpr int kTcBN = 256;
constexpr int kTcBK = 64;
constexpr int kTcStages = 4;
constexpr int kTcThreads = 192;          // producer warp, MMA warp, 4 epilogue warps
constexpr int kTcGroupM = 8;             // default tile rows per rasterisation group
constexpr int kTcEpiCols = 64;           // columns per epilogue store box
constexpr int kTcSmemBytes =
    kTcStages * (kTcBM * kTcBK + kTcBK * kTcBN) * 2   // A and B ring
    + 4 * 2 * 32 * kTcEpiCols * 2                     // 4 warps x 2 buffers x 32 x 64 x 2 B
    + 1024 /*align*/ + 256 /*barriers*/;

struct TcParams {
  int M, N, K;
  // op_a = 1: A stored K x M (an MN-major tcgen05 operand); op_b = 1: B
  // stored N x K (K-major).  The tensor maps describe the stored arrays.
  int op_a = 0, op_b = 0;
  int tiles_m, tiles_n;
  int group_m;        // tile rows per rasterisation group
  // Split-K mode (single-CTA kernel only, slices > 1): unit u is k-slice
  // u % slices of tile u / slices, stored as an FP32 partial tile at
  // ws + s * M * ldw; splitk_reduce sums the slices.  The column-split
  // fields below are unused in this mode.
  int slices;
  float* ws;
  long long ldw;
  // C := alpha * (A.B) + beta * C: the epilogue reads the old C (c_in,
  // leading dimension ldc, elements of the output type) when beta != 0.
  // Split-K units leave both to splitk_reduce.
  float alpha = 1.f, beta = 0.f;
  const void* c_in = nullptr;
  long long ldc;
  // Work units: tiles [0, full_tiles) whole (128 x 256); each later tile
  // as `parts` consecutive units of 128 x (256 / parts) columns, each over
  // the full K range.
  int full_tiles;
  int split_tiles;
  int parts;
  // Pair kernel, ksplit = 1 (parts = 2): the split tiles' units are instead
  // two ranges of K over the whole tile.  Piece 0 stores its FP32
  // accumulator at kpart (one 128 x 256 block per CTA and split tile) and
  // sets its flags to `epoch`; piece 1 waits for them, adds the partial to
  // its own accumulator, applies alpha / beta, stores C and clears the
  // flags.  kflag: one word per (split tile, CTA, epilogue warp).
  int ksplit = 0;
  float* kpart = nullptr;
  unsigned* kflag = nullptr;
  unsigned epoch = 0;
  unsigned* fault;
  unsigned long long timeout_ns;
};

// Split of an FP16/BF16 problem on `sms` persistent CTAs: the tiles of the
// last partial round (all tiles when there are fewer than `sms`) run as 2 or
// 4 narrower column parts when that many parts per tile fit in the round.
struct TcSplit {
  int split_tiles;
  int parts;
};
inline TcSplit tc_split(int tiles, int sms) {
  TcSplit sp{0, 1};
  const int rem = tiles % sms;
  if (rem == 0) return sp;
  const int fit = sms / rem;
  if (fit < 2) return sp;
  sp.split_tiles = rem;
  sp.parts = fit >= 4 ? 4 : 2;
  return sp;
}

// dtype: 1 = FP16, 2 = BF16.  tmA: A as {K, M} with 64 x 128 boxes (op_a:
// as stored {M, K}, 64 x 64 boxes); tmB: B as {N, K} with 64 x 64 boxes
// (op_b: as stored {K, N}, 64 x 64 boxes); tmC: C as {N, M} with 64 x 32
// boxes; all 128-byte swizzled.  grid = number of persistent CTAs.
cudaError_t launch_gemm_tc(int dtype, const TcParams& p, const CUtensorMap* tmA,
                           const CUtensorMap* tmB, const CUtensorMap* tmC, int grid,
                           cudaStream_t stream);

// ---------------------------------------------------------------- FP16/BF16 CTA pairs

// A cluster of two CTAs computes a 256 x 256 tile with tcgen05.mma.cta_group::2;
// each CTA stages 128 rows of A and 128 columns of B per 128-deep k-tile in a
// 3-stage ring (eight MMAs per barrier round trip).  Same 192-thread role
// layout as the single-CTA kernel.
constexpr int kTc2BM = 128;              // rows per CTA
constexpr int kTc2BN = 256;              // columns per pair tile
constexpr int kTc2BK = 128;
constexpr int kTc2Stages = 3;
constexpr int kTc2AccBufs = 2;           // accumulator buffers (256 TMEM columns each)
constexpr int kTc2SmemBytes =
    kTc2Stages * (kTc2BM * kTc2BK + kTc2BK * (kTc2BN / 2)) * 2   // A and B-half ring
    + 4 * 2 * 32 * kTcEpiCols * 2                                  // epilogue staging
    + 1024 /*align*/ + 256 /*barriers*/;

// Pair version of tc_split: the tiles of the last partial round run as two
// 128-column parts when that fits the round.
inline TcSplit tc_pair_split(int tiles, int pairs) {
  TcSplit sp{0, 1};
  const int rem = tiles % pairs;
  if (rem == 0 || 2 * rem > pairs) return sp;
  sp.split_tiles = rem;
  sp.parts = 2;
  return sp;
}

// K split of the last partial round for the pair kernel: when the leftover
// tiles fit the round twice over and K has at least kTc2KsplitMinK 128-deep
// stages, each leftover tile becomes two full-width units over two ranges
// of K; {0, 1} otherwise (the column split then applies).  Full-width units
// keep the operand feed per SM of whole tiles, where half-width column parts
// run at ~70 % of that rate.  The first range is kTc2KsplitLead stages
// shorter than half, so that the second piece's MMAs still run while the
// first stores its FP32 partial (~3.5 us, about six stages).  The hand-over
// (that store, and ~1.6 us more in the finishing epilogue) only pays for
// long K, measured on GB300: 4096^2 x 8192 FP16 174.1 -> 168.5 us, 8192^3
// BF16 593.6 -> 588 us, 4096^3 92.2 both ways, K = 2048 8-10 % slower.
constexpr int kTc2KsplitMinK = 48;
constexpr int kTc2KsplitLead = 3;
inline TcSplit tc_pair_ksplit(int tiles, int pairs, int nk) {
  TcSplit sp{0, 1};
  const int rem = tiles % pairs;
  if (rem == 0 || tiles < pairs || 2 * rem > pairs || nk < kTc2KsplitMinK) return sp;
  sp.split_tiles = rem;
  sp.parts = 2;
  return sp;
}

// 2-CTA clusters of the pair kernel (its shared memory and block size) that
// the current device can hold at once (cudaOccupancyMaxActiveClusters), or 0
// if the query fails.
int tc_pair_resident_clusters();

// tiles_m / tiles_n in p count 256 x 256 tiles; grid = 2 * pairs CTAs.
cudaError_t launch_gemm_tc_pair(int dtype, const TcParams& p, const CUtensorMap* tmA,
                                const CUtensorMap* tmB, const CUtensorMap* tmC, int pairs,
                                cudaStream_t stream);

// ---------------------------------------------------------------- split-K reduce

// C[i][j] = alpha * (sum over s of ws[s * M * ldw + i * ldw + j], in slice
// order) + beta * C[i][j], rounded once to the element type of C (elem:
// 0 = FP32, 1 = FP16, 2 = BF16); C is read only when beta != 0.  With
// c_trans, element (i, j) of C is C[j * ldc + i].
cudaError_t launch_splitk_reduce(const float* ws, int slices, int M, int N, long long ldw,
                                 void* C, long long ldc, int elem, float alpha, float beta,
                                 cudaStream_t stream, int c_trans = 0);

// D (cols x rows, row pitch ldd) := S^T for S rows x cols with row pitch lds
// (FP32): packs an operand stored transposed into the row-major layout the
// TMA-fed SGEMM reads.  D must not overlap S.
cudaError_t launch_transpose_f32(const float* S, long long rows, long long cols, long long lds,
                                 float* D, long long ldd, int sms, cudaStream_t stream);

// C := beta * C on an M x N block (C is not read when beta == 0): the
// product when K == 0 or alpha == 0.
cudaError_t launch_scale_c(void* C, int M, int N, long long ldc, int elem, float beta,
                           cudaStream_t stream);

// Split-K slice count for a grid of `tiles` output tiles over `slots` CTA
// slots and `nk` k-tiles: slices of at least 4 k-tiles, at most 32, when
// the tiles fill no more than half of the slots.
inline int splitk_slices(int tiles, int slots, int nk) {
  if (tiles <= 0 || 2 * tiles > slots) return 1;
  int s = slots / tiles;
  if (s > nk / 4) s = nk / 4;
  if (s > 32) s = 32;
  return s >= 2 ? s : 1;
}

// ---------------------------------------------------------------- shared state

// The current device's fault word (nullptr if unsupported) and the bound of
// every device-side wait, from the C-ABI translation unit.
unsigned* current_fault_word();
unsigned long long wait_bound_ns();

// Whether the GEMM kernels are launched as programmatic dependents of the
// kernel before them (DENSE_GEMM_PDL=0 turns it off, for measurement).
bool pdl_enabled();

// Launches one of the GEMM kernels (SIMT, tcgen05 single CTAs or pairs),
// which call wait_prior_grids() before their first global memory access,
// with programmatic stream serialization: its CTAs can be scheduled, and
// run their prologue (barriers, TMEM, descriptor prefetch), while the
// previous kernel in the stream finishes.  Measured on GB300, back-to-back
// FP16 GEMMs: 2048^3 18.5 -> 15.9 us, 4096^3 86.7 -> 84.4 us.
template <typename... Params, typename... Args>
cudaError_t launch_gemm_kernel(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- self test

// Waits on an mbarrier that nothing completes, with a `timeout_ns` bound; the
// wait gives up, records kFaultSelftestWait and the kernel returns.
cudaError_t launch_selftest_timeout(unsigned* fault, unsigned long long timeout_ns,
                                    cudaStream_t stream);
// Waits on a global flag that nothing sets (the K-split hand-over's wait)
// with a `timeout_ns` bound; records kFaultTcPartialWait and returns.
cudaError_t launch_selftest_flag_timeout(unsigned* fault, unsigned long long timeout_ns,
                                         cudaStream_t stream);

}  // namespace dgemm
