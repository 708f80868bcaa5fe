// FP32 SIMT SGEMM: launchers of the row-major (op N, N) kernels and the
// host copy of the shared-memory layouts.  The kernel is in sgemm_simt.cuh.
#include "sgemm_simt.cuh"

namespace dgemm {

cudaError_t launch_sgemm(const SgemmParams& p, int tn, bool use_tma, const CUtensorMap* tmA,
                         const CUtensorMap* tmB, cudaStream_t stream) {
  CUtensorMap none{};
  if (!use_tma) tmA = tmB = &none;
  if (p.op_a || p.op_b || p.c_trans) return launch_sgemm_op(p, tn, use_tma, tmA, tmB, stream);
  if (sgemm_pair_k(p.tiles_m * p.tiles_n, p.grid, p.slices)) {
    if (tn == 16)
      return use_tma ? launch_cfg<true, 16, 1, false, false, false, true>(p, tmA, tmB, stream)
                     : launch_cfg<false, 16, 1, false, false, false, true>(p, tmA, tmB, stream);
    if (tn == 9)
      return use_tma ? launch_cfg<true, 8, 1, false, false, false, true>(p, tmA, tmB, stream)
                     : launch_cfg<false, 8, 1, false, false, false, true>(p, tmA, tmB, stream);
    return use_tma ? launch_cfg<true, 8, 2, false, false, false, true>(p, tmA, tmB, stream)
                   : launch_cfg<false, 8, 2, false, false, false, true>(p, tmA, tmB, stream);
  }
  if (tn == 16)
    return use_tma ? launch_cfg<true, 16, 1>(p, tmA, tmB, stream)
                   : launch_cfg<false, 16, 1>(p, tmA, tmB, stream);
  if (tn == 9)   // 8 x 8 per thread, one CTA per SM, up to 255 registers
    return use_tma ? launch_cfg<true, 8, 1>(p, tmA, tmB, stream)
                   : launch_cfg<false, 8, 1>(p, tmA, tmB, stream);
  return use_tma ? launch_cfg<true, 8, 2>(p, tmA, tmB, stream)
                 : launch_cfg<false, 8, 2>(p, tmA, tmB, stream);
}

// Host-visible copy of the A / B stage layouts, for layout checks on the CPU.
int sgemm_smem_offset(int which, int bn, int r, int c) {
  if (which == 0) return a_tile_offset(r, c);
  return which == 1 ? b_tile_offset(bn, r, c) : bt_tile_offset(bn, r, c);
}

}  // namespace dgemm
