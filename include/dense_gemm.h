/*
 * dense_gemm.h -- C ABI of the GB300 (sm_103a) dense row-major GEMM library.
 *
 *     C[M x N] = A[M x K] . B[K x N]
 *
 * The operation is the row-major product that every page on the subject
 * starts from: "GEMM：从朴素实现到 shared memory tiling 与寄存器分块" (quant67.com)
 * states it as its computation target (row-major C_{MxN} = A_{MxK} x B_{KxN},
 * 2MNK floating-point operations), "[CUDA 优化实战] sgemm - 超越 cuBLAS"
 * (wingedge777.com) section 1 computes one C element per thread by
 * accumulating a[row*k+i] * b[i*n+col] along k, and the GB300 GEMM roadmap
 * (m.nxbn.cn) section 4.2 lays out the tensor-core form: TMA stages A and B
 * tiles in shared memory, tcgen05.mma accumulates into tensor memory, and
 * tcgen05.ld brings the result back for the epilogue.  The leading-dimension
 * arguments generalise the pages' dense layouts to row-padded ones.
 *
 * Conventions shared by every GEMM entry point:
 *  - Element (i,k) of A is A[i*lda + k]; (k,j) of B is B[k*ldb + j]; (i,j) of
 *    C is C[i*ldc + j].  Leading dimensions are in elements.
 *  - Requirements: M, N, K >= 0; lda >= K and ldb >= N when K > 0 and the
 *    operand is read; ldc >= N; A, B non-null when K > 0 and M, N > 0; C
 *    non-null when M, N > 0.  C must not overlap A or B.
 *  - M == 0 or N == 0: nothing is done and GEMM_OK is returned.  K == 0: C is
 *    set to zero (the empty sum).
 *  - C is overwritten (no alpha / beta); columns j >= N of padded C rows are
 *    never written.
 *  - Every pointer is caller-owned DEVICE memory of the current device.  The
 *    work is queued on `stream` and the call returns without synchronising.
 *  - Device memory: the library owns up to three arrays per (device,
 *    stream), each allocated by the first call that needs it and grown,
 *    after synchronising that stream, when a later call needs more; they
 *    live until the process exits and calls on different streams never
 *    share one.  (1) An FP32 workspace (gemm_plan_t.workspace_bytes, at most
 *    64 MiB): split-K slices, the FP16/BF16 pair kernel's stream-K partial
 *    tiles, and the FP32 stream-K partial tiles of scaled calls with
 *    beta != 0.  (2) An operand copy (gemm_plan_t.pack_bytes, at most
 *    1 GiB): FP32 calls with exactly one operand stored transposed, or with
 *    a row-major operand whose base or leading dimension is not 16-byte
 *    aligned (gemm_plan_t.pack).  (3) A flag array of at most 16 bytes per
 *    CTA: the hand-over flags of any grid whose tiles are cut into two
 *    pieces (gemm_plan_t.split_tiles with CTA pairs or FP32 stream-K).
 *    Calls whose plan needs none of these allocate nothing.
 *  - Accumulation is FP32 in every type.  FP16 / BF16 results are rounded to
 *    nearest-even once, from the FP32 accumulator.
 *  - Errors: argument problems are reported synchronously, before anything
 *    is queued.  A launch failure returns GEMM_ERR_LAUNCH.  A device-side
 *    wait that gave up (GEMM_ERR_DEVICE_TIMEOUT) is only visible through
 *    gemm_device_check().
 */
#ifndef DENSE_GEMM_H_
#define DENSE_GEMM_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__cplusplus)
#include <cuda_fp16.h>
#include <cuda_bf16.h>
typedef __half gemm_half_t;
typedef __nv_bfloat16 gemm_bfloat16_t;
extern "C" {
#else
/* Storage-only views of the same 16-bit formats for C callers. */
typedef struct { unsigned short bits; } gemm_half_t;     /* IEEE binary16 */
typedef struct { unsigned short bits; } gemm_bfloat16_t; /* bfloat16      */
#endif

typedef enum gemm_status_t {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_ARG = 1,        /* sizes, leading dimensions, nulls, overlap */
  GEMM_ERR_MISALIGNED = 2,         /* FP16/BF16: base or ld not 16-byte aligned */
  GEMM_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not sm_103 / no device   */
  GEMM_ERR_LAUNCH = 4,             /* the CUDA launch itself failed              */
  GEMM_ERR_DEVICE_TIMEOUT = 5,     /* a kernel's bounded wait gave up            */
  GEMM_ERR_SCRATCH_LIMIT = 6       /* gemm_f32_noalloc: problem needs more
                                      scratch than its static array holds      */
} gemm_status_t;

/*
 * FP32 GEMM on the FFMA pipes (no TF32): the SIMT kernel family of
 * wingedge777 sections 2-6 (block tiling, register outer product, swizzled
 * shared memory, coalesced write-back, multi-stage pipeline), re-designed
 * for sm_103a with a TMA-fed multi-stage ring and an 8x8 or 8x16 per-thread
 * tile chosen by problem size.
 * Any alignment is accepted: when a base pointer or lda/ldb is not 16-byte
 * aligned the operand is either copied into library scratch with 16-byte
 * rows (products of at least 2^28 multiply-adds, gemm_plan_t.pack) or its
 * tiles are staged with 4-byte cp.async instead of TMA.
 */
gemm_status_t gemm_f32(int M, int N, int K,
                       const float *A, int lda,
                       const float *B, int ldb,
                       float *C, int ldc,
                       cudaStream_t stream);

/*
 * FP16 inputs and output, FP32 accumulation, on the 5th-generation tensor
 * cores (tcgen05.mma into tensor memory, m.nxbn.cn sections 4.1-4.2).
 * A, B and C must be 16-byte aligned and lda, ldb, ldc multiples of 8
 * elements (TMA stride rule), else GEMM_ERR_MISALIGNED.
 */
gemm_status_t gemm_f16(int M, int N, int K,
                       const gemm_half_t *A, int lda,
                       const gemm_half_t *B, int ldb,
                       gemm_half_t *C, int ldc,
                       cudaStream_t stream);

/* As gemm_f16 with bfloat16 inputs and output. */
gemm_status_t gemm_bf16(int M, int N, int K,
                        const gemm_bfloat16_t *A, int lda,
                        const gemm_bfloat16_t *B, int ldb,
                        gemm_bfloat16_t *C, int ldc,
                        cudaStream_t stream);

/*
 * FP32 GEMM that never allocates device memory.  The pages have no
 * counterpart: this entry point exists for callers that cannot call
 * cudaMalloc, for example a serving process that reserves its whole memory
 * budget at start-up and may not allocate afterwards, or code whose latency
 * path cannot afford cudaMalloc's implicit synchronisation.  gemm_f32 needs
 * library-allocated memory only for split-K problems (few output tiles, long
 * K) whose slices are summed through a workspace, for stream-K grids (a
 * small array of hand-over flags) and for large products with an operand
 * TMA cannot address (re-pitched into scratch).  This variant runs the
 * same kernels but keeps the FP32 partial tiles in one fixed,
 * library-wide device array of 16 MiB and the flags in another fixed
 * array, and stages an unaligned operand with cp.async in place.
 *
 * Same arguments, conventions and results (bit for bit: the same tiles
 * and slices, summed in the same order) as gemm_f32.  A split-K problem
 * whose partial tiles need more than 16 MiB (gemm_plan_t.workspace_bytes)
 * is refused with GEMM_ERR_SCRATCH_LIMIT before anything is queued.
 *  - Set-up: the first call on a device looks up the device addresses of
 *    the arrays (cudaGetSymbolAddress), with the device current; make that
 *    first call before any stream capture.
 *  - Every call on a device shares the arrays and they keep whatever the
 *    last call wrote; nothing in them needs to start at zero (each slice
 *    is fully written before it is read; each call brings a new flag
 *    value).  Calls whose work overlaps on the GPU (different streams, no
 *    ordering between them) race on the arrays: order them, e.g. keep them
 *    on one stream.
 *  - The arrays stay allocated on every device that has loaded them until
 *    the process exits.
 */
gemm_status_t gemm_f32_noalloc(int M, int N, int K,
                               const float *A, int lda,
                               const float *B, int ldb,
                               float *C, int ldc,
                               cudaStream_t stream);

/*
 * Scaled forms: C := alpha * (A . B) + beta * C, with the conventions of
 * the plain entry points otherwise.  The m.lqnn.cn SGEMM article's tiled
 * kernel takes alpha and beta arguments (its listing leaves the beta term
 * out); the GB300 roadmap (m.nxbn.cn, section 7.1) argues for fusing such
 * epilogue work into the GEMM instead of a separate pass over C.
 *  - alpha * acc + beta * C_old is formed in FP32 (one FMA) from the FP32
 *    accumulator and rounded once to the output type.
 *  - beta == 0: the old C is not read (NaN or Inf there is ignored).
 *  - alpha == 0 or K == 0: C := beta * C and A, B are not read (they may be
 *    NULL); beta == 0 as well gives zeros.
 *  - gemm_f32_ex with beta != 0 computes the two pieces of each tile cut by
 *    the stream-K schedule into the library's workspace (two FP32 tiles per
 *    cut, gemm_plan_t.workspace_bytes) and combines them in a fixed order.
 * alpha = 1, beta = 0 is exactly the plain entry point.
 */
gemm_status_t gemm_f32_ex(int M, int N, int K, float alpha,
                          const float *A, int lda,
                          const float *B, int ldb, float beta,
                          float *C, int ldc,
                          cudaStream_t stream);
gemm_status_t gemm_f16_ex(int M, int N, int K, float alpha,
                          const gemm_half_t *A, int lda,
                          const gemm_half_t *B, int ldb, float beta,
                          gemm_half_t *C, int ldc,
                          cudaStream_t stream);
gemm_status_t gemm_bf16_ex(int M, int N, int K, float alpha,
                           const gemm_bfloat16_t *A, int lda,
                           const gemm_bfloat16_t *B, int ldb, float beta,
                           gemm_bfloat16_t *C, int ldc,
                           cudaStream_t stream);

/*
 * Storage of an operand.  The m.lqnn.cn SGEMM article (section 3.1) starts
 * from a B stored column-major, element (k, col) at B[k + col*K], and speeds
 * its kernel up by changing that layout outside the GEMM; these entry points
 * take either storage as it is:
 *   op_a == GEMM_OP_N: A stored M x K, element (i,k) at A[i*lda + k], lda >= K
 *   op_a == GEMM_OP_T: A stored K x M, element (i,k) at A[k*lda + i], lda >= M
 *   op_b == GEMM_OP_N: B stored K x N, element (k,j) at B[k*ldb + j], ldb >= N
 *   op_b == GEMM_OP_T: B stored N x K, element (k,j) at B[j*ldb + k], ldb >= K
 *                      (the article's column-major B when ldb == K)
 * C is always stored M x N row-major (ldc >= N).
 */
typedef enum gemm_op_t { GEMM_OP_N = 0, GEMM_OP_T = 1 } gemm_op_t;

/*
 * C := alpha * op(A) . op(B) + beta * C, with the conventions of the _ex
 * entry points otherwise; (GEMM_OP_N, GEMM_OP_N) is exactly gemm_*_ex.
 *  - FP16/BF16: both storages are read by TMA (a transposed A is an
 *    MN-major and a transposed B a K-major tcgen05 operand); the 16-byte
 *    alignment rule applies to lda and ldb in either storage.
 *  - FP32, exactly one operand transposed: when the product is large
 *    enough (gemm_plan_t.pack) that operand is first copied, transposed,
 *    into library scratch by an HBM-bound kernel and the row-major product
 *    runs on the copy; otherwise it is staged with 4-byte cp.async (TMA
 *    cannot transpose 4-byte elements) and the other operand by TMA when
 *    its base and leading dimension are 16-byte aligned
 *    (GEMM_PATH_SIMT_MIXED).  Any alignment is accepted either way.
 *  - FP32, both transposed: computed as C^T = B_st . A_st (two row-major
 *    arrays) with C stored transposed.
 *  - An op other than GEMM_OP_N / GEMM_OP_T is GEMM_ERR_INVALID_ARG.
 */
gemm_status_t gemm_f32_op(gemm_op_t op_a, gemm_op_t op_b, int M, int N, int K, float alpha,
                          const float *A, int lda,
                          const float *B, int ldb, float beta,
                          float *C, int ldc,
                          cudaStream_t stream);
gemm_status_t gemm_f16_op(gemm_op_t op_a, gemm_op_t op_b, int M, int N, int K, float alpha,
                          const gemm_half_t *A, int lda,
                          const gemm_half_t *B, int ldb, float beta,
                          gemm_half_t *C, int ldc,
                          cudaStream_t stream);
gemm_status_t gemm_bf16_op(gemm_op_t op_a, gemm_op_t op_b, int M, int N, int K, float alpha,
                           const gemm_bfloat16_t *A, int lda,
                           const gemm_bfloat16_t *B, int ldb, float beta,
                           gemm_bfloat16_t *C, int ldc,
                           cudaStream_t stream);

/*
 * C := alpha * op(A) . op(B) + beta * C with A, B and C in HOST memory
 * (page-locked memory lets the copies overlap the computation; pageable
 * memory works, with the copies the driver makes for it).  dtype: 0 = FP32
 * (float arrays), 1 = FP16, 2 = BF16 (16-bit arrays).  The library copies
 * B, then row blocks of A (and of C when beta != 0), into device staging
 * buffers it owns, runs each block of rows of C as a gemm_*_op call on the
 * caller's stream, and copies each block of C back as soon as it is done;
 * the copies run on two side streams of the library, so the upload of the
 * next block and the download of the previous one overlap the current
 * block's kernels.  The call returns without synchronising: the host
 * arrays must stay valid, and unmodified, until `stream` reaches this
 * point.  Work queued earlier on `stream` happens first; work queued later
 * on `stream` sees the new C.
 *  - Argument rules of gemm_*_op, except that the host arrays need no
 *    16-byte alignment (only element alignment).
 *  - Device memory: staging for A, B and C (rows padded to 16 bytes), one
 *    set per (device, stream), grown on demand after synchronising that
 *    stream, kept until the process exits; calls on one stream from several
 *    host threads are serialised on it.
 *  - Results are those of gemm_*_op on each block of rows (FP32 blocks may
 *    cut stream-K pieces elsewhere than one call on all M rows would, so
 *    the last bits can differ; integer-valued inputs give the same bits).
 */
gemm_status_t gemm_host(int dtype, gemm_op_t op_a, gemm_op_t op_b, int M, int N, int K,
                        float alpha, const void *A, int lda, const void *B, int ldb,
                        float beta, void *C, int ldc, cudaStream_t stream);
/* Row blocks gemm_host cuts an M x N product into on a GPU of num_sms SMs
 * (1, 2 or 4; blocks are multiples of 256 rows). */
int gemm_host_blocks(int dtype, int M, int N, int num_sms);
/* Ranges of K each row block of an FP32 gemm_host product runs as (1 or 3;
 * ending at ~12 % and ~40 % of K, multiples of 128, and at K): each later
 * range is a gemm_f32_op call with beta = 1 on the C the one before left,
 * so the upload before the first kernel is about an eighth as large. */
int gemm_host_k_blocks(int dtype, int M, int N, int K);

/* Static, never-null description of a status code. */
const char *gemm_status_string(gemm_status_t status);

/*
 * Synchronises `stream`, then reads and clears the current device's fault
 * word, which a kernel sets when one of its bounded waits gives up.
 * Returns GEMM_ERR_DEVICE_TIMEOUT if it was set, GEMM_ERR_LAUNCH if the
 * stream reports an error, else GEMM_OK.  *fault_bits (may be NULL)
 * receives the raw fault bits.
 */
gemm_status_t gemm_device_check(cudaStream_t stream, unsigned *fault_bits);

/*
 * Host-side plan: which kernel path a call with these arguments would take.
 * Pure host logic (no CUDA call); the dispatcher uses the same function.
 * dtype: 0 = FP32, 1 = FP16, 2 = BF16.  Pointers are only inspected for
 * alignment and overlap.  num_sms sizes persistent grids.
 */
enum {
  GEMM_PATH_NOOP = 0,          /* M == 0 or N == 0                   */
  GEMM_PATH_ZERO_FILL = 1,     /* K == 0 or alpha == 0: C := beta*C  */
  GEMM_PATH_SIMT_TMA = 2,      /* FP32 SIMT, TMA-staged tiles        */
  GEMM_PATH_SIMT_CPASYNC = 3,  /* FP32 SIMT, 4-byte cp.async tiles   */
  GEMM_PATH_TC_TMA = 4,        /* FP16/BF16 tcgen05, TMA in and out  */
  GEMM_PATH_SIMT_MIXED = 5     /* FP32 SIMT, one operand stored transposed
                                  (cp.async), the other by TMA         */
};
typedef struct gemm_plan_t {
  int path;
  int block_m, block_n, block_k, stages;
  int threads;
  int ctas;          /* grid size                         */
  int tiles;         /* output tiles                      */
  int smem_bytes;    /* dynamic shared memory per CTA     */
  int split_tiles;   /* FP32: tiles the stream-K schedule cuts into two
                        pieces (k-ranges of two CTAs); FP16/BF16: tiles
                        of the last partial round (or of a small grid)
                        run as split_pieces column parts, or, with
                        split_in_k, the tiles the stream-K share cuts    */
  int split_pieces;  /* 1 when nothing is split.  FP32: 2; the piece that
                        finishes first stores its sums to C (or, with
                        beta != 0, to a workspace tile) and the second
                        adds its own.  FP16/BF16:
                        2 or 4 column parts of the output tile, each over
                        the full K range; with split_in_k, 2 (the head
                        and the tail of a cut tile)                       */
  int cluster_ctas;  /* FP16/BF16: 2 when CTA pairs (tcgen05 cta_group::2)
                        compute 256 x 256 tiles, else 1.  FP32: 2 when the
                        two k-halves of each tile (splitk_slices = 2) run
                        as a 2-CTA cluster and add their partial tiles in
                        distributed shared memory, else 0                 */
  int splitk_slices; /* > 1: the grid is too small for the GPU, so each tile
                        is computed as this many k-slices whose FP32 partial
                        tiles go to a workspace, summed in slice order by a
                        second kernel (FP32 with cluster_ctas = 2: added
                        within the cluster, no workspace and no second
                        kernel)                                           */
  long long workspace_bytes; /* device workspace that split-K needs        */
  int pack;          /* FP32: bit 0 (A) and bit 1 (B) mark an operand
                        that is first copied by an HBM-bound kernel into
                        row-major scratch with 16-byte aligned rows (A's
                        copy first, 256-byte aligned, then B's; pack_bytes
                        in all): an operand stored transposed (exactly one
                        of the two) is transposed, a row-major one whose
                        base or leading dimension is not 16-byte aligned
                        is re-pitched.  The product then runs as the
                        row-major TMA one (path and tiles above describe
                        that run); 0 when nothing is copied               */
  long long pack_bytes;
  int split_in_k;    /* FP16/BF16 CTA pairs: 1 when the tiles from
                        streamk_first_tile on (the last partial round and
                        the round before it) are shared out among the
                        pairs as equal ranges of (tile, k-tile) work.  A
                        tile cut by a range boundary runs as a head (the
                        k-tiles before the cut, its FP32 accumulator kept
                        in the workspace) on one pair and a tail on the
                        next, whose epilogue adds that partial to its own
                        FP32 sum (in a fixed order, so results are
                        reproducible) before it stores the tile           */
  int streamk_first_tile; /* with split_in_k: first tile of the share (the
                        tiles before it run whole, in rounds)             */
} gemm_plan_t;
gemm_status_t gemm_plan(int dtype, int M, int N, int K,
                        const void *A, int lda, const void *B, int ldb,
                        const void *C, int ldc, int num_sms, gemm_plan_t *plan);
/* The plan of a scaled call (gemm_*_ex); gemm_plan is alpha = 1, beta = 0. */
gemm_status_t gemm_plan_ex(int dtype, int M, int N, int K, float alpha,
                           const void *A, int lda, const void *B, int ldb, float beta,
                           const void *C, int ldc, int num_sms, gemm_plan_t *plan);

/* The plan of a call with operand storages (gemm_*_op); gemm_plan_ex is
 * op_a = op_b = GEMM_OP_N. */
gemm_status_t gemm_plan_op(int dtype, gemm_op_t op_a, gemm_op_t op_b, int M, int N, int K,
                           float alpha, const void *A, int lda, const void *B, int ldb,
                           float beta, const void *C, int ldc, int num_sms, gemm_plan_t *plan);

/*
 * As gemm_plan_op, for a device on which only `pair_clusters` CTA pairs of
 * the FP16/BF16 pair kernel can be resident at once (0: num_sms / 2, every
 * SM; negative: GEMM_ERR_INVALID_ARG).  The pair kernel runs a persistent
 * grid of at most that many pairs.  Its K split hands an FP32 partial from
 * one pair to another, and the receiving pair polls for it; that needs
 * every pair of the grid resident together, so with fewer pairs than
 * num_sms / 2 the split is not planned.  The dispatcher plans with the
 * count cudaOccupancyMaxActiveClusters gives for the current device.
 */
gemm_status_t gemm_plan_resident(int dtype, gemm_op_t op_a, gemm_op_t op_b, int M, int N, int K,
                                 float alpha, const void *A, int lda, const void *B, int ldb,
                                 float beta, const void *C, int ldc, int num_sms,
                                 int pair_clusters, gemm_plan_t *plan);
/*
 * Inspection of a CTA-pair plan (plan->cluster_ctas == 2) for an M x N x K
 * problem: writes the work units that pair `pair` (0 <= pair < ctas / 2)
 * runs, in order, as 8 ints each -- tile row, tile column (of 256 x 256
 * tiles), first column within the tile, columns, first and end k-tile (of
 * plan->block_k), kind (0 whole, 1 head of a tile cut by the stream-K share, 2 tail
 * of one) and the range boundary of a head or tail -- up to max_units of
 * them, and returns how many units the pair runs (-1 for bad arguments).
 * Host logic only: the kernel computes the same list on the device.
 */
int gemm_pair_units(const gemm_plan_t *plan, int M, int N, int K, int pair, int *units,
                    int max_units);
/* The resident-pair count the dispatcher uses for the current device (its
 * first call on a device queries it), 0 if the query failed, -1 if there is
 * no supported device. */
int gemm_pair_clusters(void);
/* The same for the FP32 kernel's clusters over K: how many clusters of
 * `cluster_size` (2, 4 or 8) CTAs of tile configuration `config` (0 narrow
 * tiles one CTA per SM, 1 narrow two per SM, 2 wide) fit at once on the
 * current device; -1 for bad arguments or no supported device. */
int gemm_sgemm_clusters(int config, int cluster_size);

/*
 * Shared-memory layout of the kernels' operand tiles, as an element offset
 * inside one stage (for host-side bank-conflict and bijectivity checks of
 * the swizzle; wingedge777 section 4 derives its SWIZZLE_A the same way).
 * layout: 0 = FP32 A tile (128 rows x 32 k, 128-byte XOR swizzle),
 *         1 = FP32 B tile of the narrow configuration (32 k x 128 columns),
 *         2 = FP32 B tile of the wide configuration (32 k x 256 columns);
 *         these B tiles are unswizzled;
 *         3, 4 = the B tiles of the narrow / wide configuration for a B
 *         stored transposed (16-byte chunk c of row k at c ^ ((k / 4) mod 8)).
 * Returns -1 for an unknown layout or out-of-range coordinates.
 */
int gemm_smem_layout_offset(int layout, int row, int col);

/*
 * Failure-detection self test: launches one thread that waits on an
 * mbarrier nothing will complete, with a bound of `timeout_us`
 * microseconds.  The wait gives up, sets the fault word, and the kernel
 * returns; gemm_device_check() then reports GEMM_ERR_DEVICE_TIMEOUT and
 * the context stays usable.
 */
gemm_status_t gemm_selftest_timeout(unsigned timeout_us, cudaStream_t stream);
/*
 * The same for the other kind of wait: one thread polls a global flag that
 * nothing sets (the wait with which the FP16/BF16 pair kernel hands an FP32
 * partial from one K piece to the other), bounded by `timeout_us`; the
 * fault word then has bit 7 (partial never arrived) set.
 */
gemm_status_t gemm_selftest_flag_timeout(unsigned timeout_us, cudaStream_t stream);

/*
 * FP32 FFMA throughput probe: the SGEMM roofline's denominator, measured
 * rather than derived from unit counts (the m.lqnn.cn SGEMM article,
 * sections 1.1-1.2, states a kernel's efficiency against the card's FP32
 * peak).  Launches `blocks` CTAs of gemm_probe_ffma_threads() threads on
 * `stream`; each thread runs `iters` iterations of 16 independent packed
 * FMAs (fma.rn.f32x2, 4 FLOPs each) on registers only and writes one float
 * to out[block * threads + thread] (device memory, caller-owned, at least
 * blocks * threads floats).  *flops (may be NULL) receives the launch's
 * floating-point operations; the caller times the launch (CUDA events on
 * `stream`).  Non-positive sizes or a NULL out: GEMM_ERR_INVALID_ARG.
 */
gemm_status_t gemm_probe_ffma(int blocks, int iters, float *out, cudaStream_t stream,
                              double *flops);
int gemm_probe_ffma_threads(void);

#if defined(__cplusplus)
}
#endif

#endif /* DENSE_GEMM_H_ */
