// FP32 SIMT SGEMM with an operand stored transposed (A as K x M and/or B as
// N x K): the kernel of sgemm_simt.cuh with its transposing cp.async
// loaders.  A separate translation unit so that these instances compile in
// parallel with the row-major ones.
#include "sgemm_simt.cuh"

namespace dgemm {

namespace {

template <int TN, int kMinBlocks>
cudaError_t launch_ops(const SgemmParams& p, cudaStream_t stream) {
  CUtensorMap none{};
  if (p.op_a && p.op_b)
    return launch_cfg<false, TN, kMinBlocks, true, true>(p, &none, &none, stream);
  if (p.op_a) return launch_cfg<false, TN, kMinBlocks, true, false>(p, &none, &none, stream);
  return launch_cfg<false, TN, kMinBlocks, false, true>(p, &none, &none, stream);
}

}  // namespace

cudaError_t launch_sgemm_op(const SgemmParams& p, int tn, cudaStream_t stream) {
  if (tn == 16) return launch_ops<16, 1>(p, stream);
  return launch_ops<8, 2>(p, stream);
}

}  // namespace dgemm
