// Internal interface between the C-ABI dispatcher (api.cu) and the kernel
// translation units.  Not installed; callers use include/dense_gemm.h.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "dense_gemm.h"

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
// Ring stages of tile configuration tn: 16 = wide (one CTA per SM), 8 =
// narrow with two CTAs per SM, 9 = narrow with one, which has the wide
// configuration's shared memory and so twice the stages of 8.
constexpr int sgemm_stages(int tn) { return tn == 8 ? 3 : (tn == 9 ? 6 : 4); }
constexpr int sgemm_smem_bytes(int tn) {
  return sgemm_stages(tn) * (kSgemmBM * kSgemmBK + kSgemmBK * sgemm_bn(tn == 9 ? 8 : tn)) * 4 +
         1024 /*align*/ + 64 /*barriers*/;
}
// The tile configuration of a kernel instance: TN outputs per thread row,
// kMinBlocks CTAs per SM.
constexpr int sgemm_cfg(int tn, int min_blocks) { return tn == 8 && min_blocks == 1 ? 9 : tn; }

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
  // split_tiles tiles are cut by a range boundary into two pieces, which
  // meet through boundary c's words sk_flags[2 (c - 1)] (arrival: the
  // first piece to finish finds a value other than epoch there) and
  // sk_flags[2 (c - 1) + 1] (done: set to epoch once the first piece's
  // result is visible).  With tail_ws == nullptr (only when beta = 0) the
  // first piece stores alpha times its FP32 sums to C and the second adds
  // alpha times its own into it; otherwise the first stores its unscaled
  // sums at tail_ws + (c - 1) * BM * BN (row-major, leading dimension BN)
  // and the second writes alpha * (sum + sum) + beta * C.  With exactly two
  // addends the result does not depend on which piece came first.  Each
  // launch brings a new epoch, and the second piece clears both words once
  // it has seen the first's, so a replayed launch (same epoch) works too.
  int grid;
  int dp_tiles = 0;
  int split_tiles;
  float* tail_ws = nullptr;
  unsigned* sk_flags = nullptr;   // 2 (grid - 1) words when split_tiles > 0
  unsigned epoch = 0;             // non-zero, new for every launch
  // Split-K mode (slices > 1): CTA u computes k-slice u % slices of tile
  // u / slices (k-tiles [s*nk/slices, (s+1)*nk/slices)) and stores its FP32
  // partial tile at ws + s * M * ldw (row-major, leading dimension ldw);
  // splitk_reduce then sums the slices in slice order into C.  grid and
  // split_tiles are unused in this mode.
  int slices;
  float* ws;
  long long ldw;
  // cluster_k = 1 (slices == 1, grid = 2 tiles, dp_tiles = 0): CTAs 2t and
  // 2t + 1 compute tile t over the two halves of K as a cluster of two and
  // add their halves in distributed shared memory; no flags, no workspace.
  int cluster_k = 0;
  // C := alpha * (A.B) + beta * C; the old C is read only when beta != 0
  // (in split-K mode splitk_reduce applies alpha and beta; for a cut tile
  // the piece that completes it does).
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
// zero fill.  Returns the launch error.
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
  // C's columns [0, n_tma) go out through TMA stores (tmC's inner extent is
  // n_tma: N rounded down to a multiple of 8 elements, since a TMA store
  // whose clipped edge falls inside a 16-byte granule writes the whole
  // granule); the ragged tail [n_tma, N) through plain 2-byte stores to
  // c_out.  n_tma == 0 (N < 8): no TMA stores at all.
  int n_tma = 0;
  void* c_out = nullptr;
  // Work units: tiles [0, full_tiles) whole (128 x 256); each later tile
  // as `parts` consecutive units of 128 x (256 / parts) columns, each over
  // the full K range.
  int full_tiles;
  int split_tiles;
  int parts;
  // Pair kernel, sk = 1 (stream-K share): tiles [0, sk_first_tile) run as
  // whole tiles in rounds of the grid's pairs, and the sk_tiles tiles after
  // them are shared out as equal ranges of (tile, k-tile) steps, one range
  // per pair (sk_tiles >= pairs, so a tile is cut at most once).  The head
  // of a cut tile (k-tiles before the cut) stores its FP32 accumulator at
  // kpart (one 128 x 256 block per CTA and range boundary) and sets its
  // flags to `epoch`; the pair running the tail waits for them in its last
  // epilogue, adds the partial to its own accumulator, then clears the
  // flags.  kflag: one word per (range boundary, CTA, epilogue warp).
  // full_tiles, split_tiles and parts are unused in this mode.
  int sk = 0;
  int sk_first_tile = 0;
  int sk_tiles = 0;
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
// Tile rows (of 256) per rasterisation group: measured on GB300, 4096^3 FP16
// 86.7 us with 16 against 88.7 with 8 (4 and 6 no better), 8192^3 BF16 the
// same with 8 or 16.
constexpr int kTc2GroupM = 16;
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

// Stream-K share of the pair kernel (TcParams::sk): when the tiles do not
// fill whole rounds of `pairs`, the last partial round and the round before
// it (or the two rounds before it) are shared out as equal ranges of
// (tile, k-tile) steps instead of running as a partial round.  A range is
// then share = R nk / P k-tiles for R shared tiles, and a tail ends at
// least share - nk k-tiles after the head it needs: the one round is taken
// when that leaves kTc2StreamkSlack k-tiles for the head's partial to be
// stored (about 4 us), else two.  Needs at least kTc2StreamkMinK k-tiles
// per tile: measured on GB300 against the partial round (column parts),
// 4096^2 x K FP16: K = 8192 164.5 vs 174.8 us, 4096 90.8 vs 93.9, 2048
// 54.0 vs 53.9, 1024 39.6 vs 33.4; BF16 4097 x 3000 x 1536 43.7 vs 39.6.  Returns the first tile of the share (a multiple of pairs), or
// -1 for no share.
constexpr int kTc2StreamkMinK = 3072 / kTc2BK;
constexpr int kTc2StreamkSlack = 1024 / kTc2BK;
inline int tc_pair_streamk_first(int tiles, int pairs, int nk, int min_rounds = 1) {
  if (pairs < 2 || tiles < pairs || tiles % pairs == 0 || nk < kTc2StreamkMinK) return -1;
  for (int r = min_rounds; r <= 2 && tiles / pairs >= r; ++r) {
    const int first = (tiles / pairs - r) * pairs;
    const long long slack = (long long)(tiles - first - pairs) * nk / pairs;
    if (slack >= kTc2StreamkSlack) return first;
  }
  return -1;
}

// Tiles a stream-K share of `tiles` tiles (>= pairs) of nk k-tiles over
// `pairs` ranges cuts: boundaries q * tiles * nk / pairs, q = 1 .. pairs - 1,
// that fall inside a tile (the kernel's rule).
inline int tc_pair_streamk_cuts(int tiles, int pairs, int nk) {
  const long long total = (long long)tiles * nk;
  int cuts = 0;
  for (int q = 1; q < pairs; ++q)
    if (((long long)q * total / pairs) % nk != 0) ++cuts;
  return cuts;
}

// Work unit of the pair-persistent grid: 256 x 256 tile (tm, tn), the
// columns [n_off, n_off + n_w) of it (all 256, or one of two 128-column
// parts of a tile of a last partial round) and the k-tiles [kb, ke).
//
// Two schedules (TcParams::sk):
//  * sk = 0: pair q computes units q, q + P, q + 2P, ... of the unit list
//    (whole tiles, then the column parts of the split tiles), P pairs;
//  * sk = 1 (stream-K share): tiles [0, D) (D = sk_first_tile, a multiple of
//    P) are whole units in rounds of P, pair q taking q, q + P, ...; the
//    R = sk_tiles tiles after them are one iteration space of R * nk
//    (tile, k-tile) steps, of which pair q takes the steps
//    [q R nk / P, (q + 1) R nk / P) -- at least one tile's worth, since
//    R >= P, so a range boundary cuts a tile at most once.  A cut tile is
//    two units: its head (k-tiles [0, h)) on the pair whose range ends
//    inside it, and its tail (k-tiles [h, nk)) on the next pair.  A pair
//    runs its whole tiles of the rounds first (all pairs in step, so that
//    the rounds' operands are shared in L2), then its head, which stores
//    the FP32 accumulator to the workspace and raises a flag, then the
//    whole tiles of its range, and its tail last: the tail's epilogue adds
//    the previous pair's head partial (stored one share earlier) to its own
//    accumulator, in that fixed order, and finishes the tile.
constexpr int kTcUnitWhole = 0, kTcUnitHead = 1, kTcUnitTail = 2;
struct TcUnit {
  int tm, tn, n_off, n_w, kb, ke;
  int kind;    // kTcUnitWhole, kTcUnitHead or kTcUnitTail
  int slot;    // head / tail: the range boundary that cuts the tile (1 .. P - 1)
};

// The units of one pair, in the order it runs them.
struct TcPairSched {
  int n;                   // number of units
  int has_head, has_tail;  // stream-K: unit nd is a head, unit n - 1 a tail
  int nd;                  // stream-K: whole tiles of the rounds before the share
  int w0, nw;              // stream-K: whole tiles [w0, w0 + nw) of the share
  int head_tile, head_ke, tail_tile, tail_kb;
  int pair;
};
__host__ __device__ inline TcPairSched tc_pair_sched(int pair, int npairs, const TcParams& p,
                                                     int nk) {
  TcPairSched s;
  s.pair = pair;
  s.has_head = s.has_tail = 0;
  s.nd = s.w0 = s.nw = 0;
  s.head_tile = s.head_ke = s.tail_tile = s.tail_kb = 0;
  if (!p.sk) {
    const int num_units = p.full_tiles + p.split_tiles * p.parts;
    s.n = pair < num_units ? (num_units - pair + npairs - 1) / npairs : 0;
    return s;
  }
  const long long total = (long long)p.sk_tiles * nk;
  const long long b = (long long)pair * total / npairs;
  const long long e = (long long)(pair + 1) * total / npairs;
  s.has_head = (e % nk) != 0;
  s.has_tail = (b % nk) != 0;
  s.nd = p.sk_first_tile / npairs;
  const int first_whole = (int)((b + nk - 1) / nk);
  s.w0 = p.sk_first_tile + first_whole;
  s.nw = (int)(e / nk) - first_whole;
  s.head_tile = p.sk_first_tile + (int)(e / nk);
  s.head_ke = (int)(e % nk);
  s.tail_tile = p.sk_first_tile + (int)(b / nk);
  s.tail_kb = (int)(b % nk);
  s.n = s.has_head + s.nd + s.nw + s.has_tail;
  return s;
}

// Unit j (0 <= j < s.n) of the pair that s describes.
__host__ __device__ inline TcUnit tc_pair_unit(const TcPairSched& s, int j, int npairs,
                                               const TcParams& p, int nk) {
  TcUnit w;
  int tile;
  w.n_off = 0;
  w.n_w = kTc2BN;
  w.kb = 0;
  w.ke = nk;
  w.kind = kTcUnitWhole;
  w.slot = 0;
  if (!p.sk) {
    const int u = s.pair + j * npairs;
    if (u < p.full_tiles) {
      tile = u;
    } else {
      const int i = u - p.full_tiles;
      tile = p.full_tiles + i / p.parts;
      w.n_w = kTc2BN / p.parts;
      w.n_off = (i % p.parts) * w.n_w;
    }
  } else if (j < s.nd) {
    tile = s.pair + j * npairs;
  } else if (s.has_head && j == s.nd) {
    tile = s.head_tile;
    w.ke = s.head_ke;
    w.kind = kTcUnitHead;
    w.slot = s.pair + 1;
  } else {
    const int i = j - s.nd - s.has_head;
    if (i < s.nw) {
      tile = s.w0 + i;
    } else {
      tile = s.tail_tile;
      w.kb = s.tail_kb;
      w.kind = kTcUnitTail;
      w.slot = s.pair;
    }
  }
  grouped_tile(tile, p.tiles_m, p.tiles_n, p.group_m, w.tm, w.tn);
  return w;
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

// One re-pitch copy: D (rows x cols, row pitch ldd, a multiple of 4,
// 16-byte aligned) := S (row pitch lds, any 4-byte alignment), FP32; the
// padding columns of D are zeroed.  D must not overlap S.
struct RepitchJob {
  const float* S;
  long long rows, cols, lds;
  float* D;
  long long ldd;
};

// Re-pitches 1 or 2 operands whose rows TMA cannot address, in one launch.
cudaError_t launch_repitch_f32(const RepitchJob* jobs, int njobs, int sms, cudaStream_t stream);
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

// Caller-owned device scratch for an FP32 call that must not allocate:
// `flag_words` flag words for the stream-K hand-over (SgemmParams::
// sk_flags; written by nothing but the GEMM kernels), the launch's epoch
// (non-zero, new for every launch that uses them), and `ws_bytes` of FP32
// split-K workspace.
struct FixedScratch {
  unsigned* flags;
  long long flag_words;
  unsigned epoch;
  float* ws;
  long long ws_bytes;
};

// gemm_f32 that allocates nothing: no operand is copied into scratch (an
// unaligned row-major operand is staged by 4-byte cp.async) and the flags
// and workspace come from `scratch` (GEMM_ERR_SCRATCH_LIMIT, before
// anything is queued, if they are too small).
gemm_status_t run_f32_no_copy(int M, int N, int K, const float* A, int lda, const float* B,
                              int ldb, float* C, int ldc, cudaStream_t stream,
                              const FixedScratch& scratch);

// 2-, 4- and 8-CTA clusters of the SGEMM kernel that fit on the current
// device at once, n[cfg][0 / 1 / 2] for s = 2 / 4 / 8, cfg 0 = narrow
// tiles with one CTA per SM, 1 = narrow with two, 2 = wide
// (cudaOccupancyMaxActiveClusters; 0 where the query failed).
struct SgemmClusterCaps {
  int n[3][3];
};
SgemmClusterCaps sgemm_cluster_caps();

// Whether the GEMM kernels are launched as programmatic dependents of the
// kernel before them (DENSE_GEMM_PDL=0 turns it off, for measurement).
bool pdl_enabled();

// Launches one of the GEMM kernels (SIMT, tcgen05 single CTAs or pairs),
// which call wait_prior_grids() before their first global memory access,
// with programmatic stream serialization: its CTAs can be scheduled, and
// run their prologue (barriers, TMEM, descriptor prefetch), while the
// previous kernel in the stream finishes.  Measured on GB300, back-to-back
// FP16 GEMMs: 2048^3 18.5 -> 15.9 us, 4096^3 86.7 -> 84.4 us.  cluster_x > 1
// groups consecutive CTAs into clusters of that many (a kernel compiled
// with __cluster_dims__ takes 1 here).
template <typename... Params, typename... Args>
cudaError_t launch_gemm_kernel_clusters(unsigned cluster_x, void (*kernel)(Params...), dim3 grid,
                                        dim3 block, size_t smem, cudaStream_t stream,
                                        Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... Params, typename... Args>
cudaError_t launch_gemm_kernel(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, Args&&... args) {
  return launch_gemm_kernel_clusters(1, kernel, grid, block, smem, stream,
                                     std::forward<Args>(args)...);
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
