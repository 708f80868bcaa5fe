// gemm_host: the product on operands and result in host memory.  The
// library copies them to device staging buffers it owns and overlaps the
// copies with the computation: C is cut into row blocks, and a large FP32
// product also into ranges of K; while the GEMM of one block runs on
// the caller's stream, the operands of the next go up on one side stream
// and the finished rows of C come back on another.  Each block is an
// ordinary gemm_*_op call on device memory (a later K range with beta = 1
// on the C the earlier one left), so every block takes the same kernels and
// planning as a device call of its shape.
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include <cuda_runtime.h>

#include "dense_gemm.h"

namespace {

constexpr int kMaxBlocks = 4;    // row blocks
constexpr int kMaxKBlocks = 3;   // ranges of K (FP32)
// Ends of the ranges of K, in percent of K (rounded up to 128): a short
// first range, so that the first kernel waits for little of A and B, each
// later range long enough for the kernel before it to outlast its upload.
// Measured on GB300, 4096^3 FP32 through gemm_host alone / with the FP16
// 4096^3 problem on a second stream: ranges ending at 35 % and 100 %
// 2.51 / 2.77 ms; 25 / 100 2.47 / 2.69; 20 / 100 2.52 / 2.77; 15 / 100
// 2.61 / 2.83; 15 / 45 / 100 2.46 / 2.69; 10 / 35 / 100 2.44 / 2.66-2.69;
// 8 / 30 / 100 2.43 / 2.62-2.67; 10 / 30 / 100 2.45 / 2.65-2.67;
// 12 / 40 / 100 2.43 / 2.61-2.63.
constexpr int kKEndPct[kMaxKBlocks] = {12, 40, 100};
constexpr int kKRanges = 3;
constexpr int kRowAlign = 256;   // row blocks are whole CTA-pair tile rows

struct HostStaging {
  void* a = nullptr;
  void* b = nullptr;
  void* c = nullptr;
  size_t a_bytes = 0, b_bytes = 0, c_bytes = 0;
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t in[kMaxBlocks * kMaxKBlocks] = {}, out[kMaxBlocks] = {};
  std::mutex mu;   // one enqueue at a time per (device, stream)
};

std::mutex g_host_mu;
std::map<std::pair<int, cudaStream_t>, HostStaging*> g_host;   // guarded by g_host_mu

bool ok(cudaError_t e) {
  if (e == cudaSuccess) return true;
  cudaGetLastError();
  return false;
}

gemm_status_t staging_for(cudaStream_t stream, HostStaging** out) {
  int dev = -1;
  if (!ok(cudaGetDevice(&dev))) return GEMM_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_host_mu);
  HostStaging*& h = g_host[std::make_pair(dev, stream)];
  if (h == nullptr) {
    HostStaging* n = new HostStaging;
    bool good = ok(cudaStreamCreateWithFlags(&n->up, cudaStreamNonBlocking)) &&
                ok(cudaStreamCreateWithFlags(&n->down, cudaStreamNonBlocking)) &&
                ok(cudaEventCreateWithFlags(&n->start, cudaEventDisableTiming)) &&
                ok(cudaEventCreateWithFlags(&n->done, cudaEventDisableTiming));
    for (int i = 0; good && i < kMaxBlocks * kMaxKBlocks; ++i)
      good = ok(cudaEventCreateWithFlags(&n->in[i], cudaEventDisableTiming));
    for (int i = 0; good && i < kMaxBlocks; ++i)
      good = ok(cudaEventCreateWithFlags(&n->out[i], cudaEventDisableTiming));
    if (!good) {
      delete n;   // (any streams or events made are left to process exit)
      g_host.erase(std::make_pair(dev, stream));
      return GEMM_ERR_LAUNCH;
    }
    h = n;
  }
  *out = h;
  return GEMM_OK;
}

// Grows one staging buffer; earlier calls queued on the stream may still use
// the old one, so the stream and both side streams are drained first.
bool reserve(HostStaging* h, cudaStream_t stream, void** buf, size_t* have, size_t need) {
  if (*have >= need) return true;
  if (*buf != nullptr) {
    if (!ok(cudaStreamSynchronize(stream)) || !ok(cudaStreamSynchronize(h->up)) ||
        !ok(cudaStreamSynchronize(h->down)))
      return false;
    cudaFree(*buf);
    *buf = nullptr;
    *have = 0;
  }
  if (!ok(cudaMalloc(buf, need))) {
    *buf = nullptr;
    return false;
  }
  *have = need;
  return true;
}

inline long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }

// Bytes spanned by a rows x cols array with row pitch ld, and whether two
// byte ranges intersect.
inline uint64_t span(long long rows, long long cols, long long ld, size_t es) {
  return rows <= 0 || cols <= 0 ? 0 : (uint64_t)((rows - 1) * ld + cols) * es;
}
inline bool overlaps(const void* a, uint64_t an, const void* b, uint64_t bn) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return an != 0 && bn != 0 && a0 < b0 + bn && b0 < a0 + an;
}

gemm_status_t run_device(int dtype, int op_a, int op_b, int M, int N, int K, float alpha,
                         const void* A, int lda, const void* B, int ldb, float beta, void* C,
                         int ldc, cudaStream_t stream) {
  const gemm_op_t oa = op_a ? GEMM_OP_T : GEMM_OP_N, ob = op_b ? GEMM_OP_T : GEMM_OP_N;
  if (dtype == 0)
    return gemm_f32_op(oa, ob, M, N, K, alpha, static_cast<const float*>(A), lda,
                       static_cast<const float*>(B), ldb, beta, static_cast<float*>(C), ldc,
                       stream);
  if (dtype == 1)
    return gemm_f16_op(oa, ob, M, N, K, alpha, static_cast<const gemm_half_t*>(A), lda,
                       static_cast<const gemm_half_t*>(B), ldb, beta,
                       static_cast<gemm_half_t*>(C), ldc, stream);
  return gemm_bf16_op(oa, ob, M, N, K, alpha, static_cast<const gemm_bfloat16_t*>(A), lda,
                      static_cast<const gemm_bfloat16_t*>(B), ldb, beta,
                      static_cast<gemm_bfloat16_t*>(C), ldc, stream);
}

}  // namespace

extern "C" int gemm_host_blocks(int dtype, int M, int N, int num_sms) {
  if (M <= 0 || N <= 0) return 1;
  // FP32 is compute-bound at any size that is worth splitting: two blocks,
  // each still a full grid of 128 x 256 tiles.  FP16 / BF16 move twice as
  // many bytes per FLOP through the copies as they spend computing, so four
  // blocks overlap more of the download with the uploads.
  const int sms = num_sms > 0 ? num_sms : 1;
  for (int nb = dtype == 0 ? 2 : kMaxBlocks; nb > 1; nb /= 2) {
    const long long rows = round_up((M + nb - 1) / nb, kRowAlign);
    if (rows * (nb - 1) >= M) continue;   // the last block would be empty
    if (dtype == 0 && ((rows + 127) / 128) * ((N + 255) / 256) < sms) continue;
    return nb;
  }
  return 1;
}

extern "C" int gemm_host_k_blocks(int dtype, int M, int N, int K) {
  // FP32 only: the partial C between ranges stays FP32, where FP16 / BF16
  // would round it to 16 bits once more.  kKRanges ranges of K (ending at
  // kKEndPct percent of K) when the product is large enough (>= 2^36
  // FLOPs) for the shorter first upload to matter against the extra
  // launches and smaller grids.
  if (dtype != 0 || K < 2048 || M <= 0 || N <= 0) return 1;
  return 2.0 * M * N * K >= 68719476736.0 ? kKRanges : 1;
}

extern "C" gemm_status_t gemm_host(int dtype, gemm_op_t op_a, gemm_op_t op_b, int M, int N,
                                   int K, float alpha, const void* A, int lda, const void* B,
                                   int ldb, float beta, void* C, int ldc, cudaStream_t stream) {
  // The device entry points' argument rules, on the host arrays; the host
  // arrays need no 16-byte alignment (the staging copies have it).
  if (dtype < 0 || dtype > 2) return GEMM_ERR_INVALID_ARG;
  if ((op_a != GEMM_OP_N && op_a != GEMM_OP_T) || (op_b != GEMM_OP_N && op_b != GEMM_OP_T))
    return GEMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  const size_t es = dtype == 0 ? 4 : 2;
  if (C == nullptr || ldc < N || reinterpret_cast<uintptr_t>(C) % es) return GEMM_ERR_INVALID_ARG;
  const bool reads_ab = K > 0 && alpha != 0.f;   // else C := beta * C
  // Stored shapes (rows x cols): A is M x K or K x M, B is K x N or N x K.
  const long long a_rows = op_a ? K : M, a_cols = op_a ? M : K;
  const long long b_rows = op_b ? N : K, b_cols = op_b ? K : N;
  if (reads_ab) {
    if (A == nullptr || B == nullptr || lda < a_cols || ldb < b_cols ||
        reinterpret_cast<uintptr_t>(A) % es || reinterpret_cast<uintptr_t>(B) % es)
      return GEMM_ERR_INVALID_ARG;
    if (overlaps(A, span(a_rows, a_cols, lda, es), C, span(M, N, ldc, es)) ||
        overlaps(B, span(b_rows, b_cols, ldb, es), C, span(M, N, ldc, es)))
      return GEMM_ERR_INVALID_ARG;
  }
  gemm_status_t st = GEMM_OK;
  int dev = -1, sms = 0;
  if (!ok(cudaGetDevice(&dev)) ||
      !ok(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)))
    return GEMM_ERR_UNSUPPORTED_DEVICE;
  HostStaging* h = nullptr;
  st = staging_for(stream, &h);
  if (st != GEMM_OK) return st;
  std::lock_guard<std::mutex> lock(h->mu);

  const long long pad = 16 / (long long)es;   // device rows start 16-byte aligned
  const bool reads_c = beta != 0.f;
  const long long dla = round_up(a_cols, pad), dlb = round_up(b_cols, pad);
  const long long dlc = round_up(N, pad);
  if ((reads_ab && (!reserve(h, stream, &h->a, &h->a_bytes, (size_t)(a_rows * dla) * es) ||
                    !reserve(h, stream, &h->b, &h->b_bytes, (size_t)(b_rows * dlb) * es))) ||
      !reserve(h, stream, &h->c, &h->c_bytes, (size_t)((long long)M * dlc) * es))
    return GEMM_ERR_LAUNCH;

  const int nb = gemm_host_blocks(dtype, M, N, sms);
  // Row block i is rows [start(i), start(i + 1)), block boundaries whole
  // 256-row units.  FP16 / BF16: equal blocks.  FP32 (two blocks): the last
  // as small as still gives every SM a 128 x 256 tile, so the least of C is
  // left to download after the last kernel (4096^2: 2816 + 1280 rows).
  const int rows = nb == 1 ? M : (int)round_up((M + nb - 1) / nb, kRowAlign);
  int split = rows;   // FP32, two blocks: the first row of the second
  if (dtype == 0 && nb == 2) {
    const int tiles_n = (N + 255) / 256;
    const long long need = round_up((long long)((sms + tiles_n - 1) / tiles_n) * 128, kRowAlign);
    if (need < M - rows) split = (int)((M - need) / kRowAlign * kRowAlign);
  }
  const auto start = [&](int i) {
    if (dtype == 0 && nb == 2) return i == 0 ? 0 : (i == 1 ? split : M);
    const long long r = (long long)i * rows;
    return r < M ? (int)r : M;
  };
  const int nkb = reads_ab ? gemm_host_k_blocks(dtype, M, N, K) : 1;
  // Range j of K is [kend(j - 1), kend(j)).
  const auto kend = [&](int j) {
    if (j >= nkb - 1) return K;
    const long long e = round_up((long long)K * kKEndPct[j] / 100, 128);
    return e < K ? (int)e : K;
  };
  unsigned char* const da = static_cast<unsigned char*>(h->a);
  unsigned char* const db = static_cast<unsigned char*>(h->b);
  unsigned char* const dc = static_cast<unsigned char*>(h->c);
  const unsigned char* const ha = static_cast<const unsigned char*>(A);
  const unsigned char* const hb = static_cast<const unsigned char*>(B);
  unsigned char* const hc = static_cast<unsigned char*>(C);
  const auto up = [&](void* dst, size_t dpitch, const void* src, size_t spitch, size_t width,
                       size_t height) {
    return width == 0 || height == 0 ||
           ok(cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, height,
                                cudaMemcpyHostToDevice, h->up));
  };

  // Everything queued before this call on `stream` happens first.
  if (!ok(cudaEventRecord(h->start, stream)) || !ok(cudaStreamWaitEvent(h->up, h->start, 0)) ||
      !ok(cudaStreamWaitEvent(h->down, h->start, 0)))
    return GEMM_ERR_LAUNCH;
  for (int i = 0; i < nb; ++i) {
    const int r0 = start(i);
    const int m = start(i + 1) - r0;
    unsigned char* c_dev = dc + (size_t)r0 * dlc * es;
    unsigned char* c_host = hc + (size_t)r0 * ldc * es;
    for (int j = 0; j < nkb; ++j) {
      const int k0 = j == 0 ? 0 : kend(j - 1);
      const int kk = kend(j) - k0;
      if (j > 0 && kk <= 0) continue;   // (a range that rounding left empty)
      // B's rows k0.. (stored K x N) or columns k0.. (stored N x K), once.
      unsigned char* b_blk = op_b ? db + (size_t)k0 * es : db + (size_t)k0 * dlb * es;
      if (reads_ab && i == 0) {
        const unsigned char* b_src = op_b ? hb + (size_t)k0 * es : hb + (size_t)k0 * ldb * es;
        if (!up(b_blk, dlb * es, b_src, (size_t)ldb * es,
                (op_b ? (size_t)kk : (size_t)N) * es, op_b ? (size_t)N : (size_t)kk))
          return GEMM_ERR_LAUNCH;
      }
      // A's rows r0.. and columns k0.. (stored M x K), or rows k0.. and
      // columns r0.. (stored K x M).
      const size_t a_off = op_a ? (size_t)k0 * dla + r0 : (size_t)r0 * dla + k0;
      unsigned char* a_blk = da + a_off * es;
      if (reads_ab) {
        const size_t h_off = op_a ? (size_t)k0 * lda + r0 : (size_t)r0 * lda + k0;
        if (!up(a_blk, dla * es, ha + h_off * es, (size_t)lda * es,
                (op_a ? (size_t)m : (size_t)kk) * es, op_a ? (size_t)kk : (size_t)m))
          return GEMM_ERR_LAUNCH;
      }
      if (j == 0 && reads_c &&
          !up(c_dev, dlc * es, c_host, (size_t)ldc * es, (size_t)N * es, (size_t)m))
        return GEMM_ERR_LAUNCH;
      cudaEvent_t in = h->in[i * kMaxKBlocks + j];
      if (!ok(cudaEventRecord(in, h->up)) || !ok(cudaStreamWaitEvent(stream, in, 0)))
        return GEMM_ERR_LAUNCH;
      // A later range of K adds onto the C the earlier one left.
      st = run_device(dtype, op_a, op_b, m, N, reads_ab ? kk : K, alpha,
                      reads_ab ? a_blk : nullptr, (int)dla, reads_ab ? b_blk : nullptr, (int)dlb,
                      j == 0 ? beta : 1.f, c_dev, (int)dlc, stream);
      if (st != GEMM_OK) return st;
    }
    if (!ok(cudaEventRecord(h->out[i], stream)) ||
        !ok(cudaStreamWaitEvent(h->down, h->out[i], 0)) ||
        !ok(cudaMemcpy2DAsync(c_host, (size_t)ldc * es, c_dev, dlc * es, (size_t)N * es, m,
                              cudaMemcpyDeviceToHost, h->down)))
      return GEMM_ERR_LAUNCH;
  }
  // The call is complete, in stream order, once the last rows are back.
  if (!ok(cudaEventRecord(h->done, h->down)) || !ok(cudaStreamWaitEvent(stream, h->done, 0)))
    return GEMM_ERR_LAUNCH;
  return GEMM_OK;
}
