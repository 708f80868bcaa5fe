// FP32 SIMT SGEMM: launchers of the row-major (op N, N) kernels and the
// host copy of the shared-memory layouts.  The kernel is in sgemm_simt.cuh.
#include "sgemm_simt.cuh"

namespace dgemm {

cudaError_t launch_sgemm(const SgemmParams& p, int tn, bool use_tma, const CUtensorMap* tmA,
                         const CUtensorMap* tmB, cudaStream_t stream) {
  CUtensorMap none{};
  if (!use_tma) tmA = tmB = &none;
  if (p.op_a || p.op_b || p.c_trans) return launch_sgemm_op(p, tn, use_tma, tmA, tmB, stream);
  if (p.cluster_k) {
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

namespace {

template <bool kTma, int TN, int kMinBlocks>
int cluster_capacity(int s) {
  const auto kernel = sgemm_kernel<kTma, TN, kMinBlocks, false, false, false, true>;
  constexpr int kSmem = sgemm_smem_bytes(sgemm_cfg(TN, kMinBlocks));
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)s);
  cfg.blockDim = dim3(kSgemmThreads);
  cfg.dynamicSmemBytes = kSmem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = (unsigned)s;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return clusters;
}

}  // namespace

SgemmClusterCaps sgemm_cluster_caps() {
  // The TMA instances stand for the cp.async ones: same block and shared
  // memory, and both keep the CTAs per SM that their launch bounds name.
  SgemmClusterCaps c{};
  const int sizes[3] = {2, 4, 8};
  for (int i = 0; i < 3; ++i) {
    c.n[0][i] = cluster_capacity<true, 8, 1>(sizes[i]);
    c.n[1][i] = cluster_capacity<true, 8, 2>(sizes[i]);
    c.n[2][i] = cluster_capacity<true, 16, 1>(sizes[i]);
  }
  return c;
}

// Host-visible copy of the A / B stage layouts, for layout checks on the CPU.
int sgemm_smem_offset(int which, int bn, int r, int c) {
  if (which == 0) return a_tile_offset(r, c);
  return which == 1 ? b_tile_offset(bn, r, c) : bt_tile_offset(bn, r, c);
}

}  // namespace dgemm
