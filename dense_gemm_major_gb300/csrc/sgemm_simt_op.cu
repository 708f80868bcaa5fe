// FP32 SIMT SGEMM with an operand stored transposed (A as K x M and/or B as
// N x K): the kernel of sgemm_simt.cuh with its transposing cp.async
// loaders, the other operand by TMA where it is 16-byte aligned; and the
// row-major kernel that stores C transposed (the product of two operands
// both stored transposed is computed as C^T).  A separate translation unit so that these instances compile in
// parallel with the row-major ones.
#include "sgemm_simt.cuh"

namespace dgemm {

namespace {

template <int TN, int kMinBlocks>
cudaError_t launch_ops(const SgemmParams& p, bool use_tma, const CUtensorMap* tmA,
                       const CUtensorMap* tmB, cudaStream_t stream) {
  if (p.c_trans)   // row-major operands, C stored transposed
    return use_tma ? launch_cfg<true, TN, kMinBlocks, false, false, true>(p, tmA, tmB, stream)
                   : launch_cfg<false, TN, kMinBlocks, false, false, true>(p, tmA, tmB, stream);
  if (p.op_a && p.op_b) return launch_cfg<false, TN, kMinBlocks, true, true>(p, tmA, tmB, stream);
  if (p.op_a)
    return use_tma ? launch_cfg<true, TN, kMinBlocks, true, false>(p, tmA, tmB, stream)
                   : launch_cfg<false, TN, kMinBlocks, true, false>(p, tmA, tmB, stream);
  return use_tma ? launch_cfg<true, TN, kMinBlocks, false, true>(p, tmA, tmB, stream)
                 : launch_cfg<false, TN, kMinBlocks, false, true>(p, tmA, tmB, stream);
}

}  // namespace

cudaError_t launch_sgemm_op(const SgemmParams& p, int tn, bool use_tma, const CUtensorMap* tmA,
                            const CUtensorMap* tmB, cudaStream_t stream) {
  if (tn == 16) return launch_ops<16, 1>(p, use_tma, tmA, tmB, stream);
  return launch_ops<8, 2>(p, use_tma, tmA, tmB, stream);
}

}  // namespace dgemm
