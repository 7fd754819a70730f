// Tensor-core contractions with a plain scaled store: dH = (dloss/N) G W and
// dW (+)= (dloss/N) G^T h of the backward, and the building-block GEMM the
// tests use to check every operand layout.
#include "lce_device.cuh"

namespace lce {

cudaError_t launch_gemm_store(bool a_mn, bool b_mn, const CUtensorMap& ta,
                              const CUtensorMap& tb, const GemmGeom& g,
                              const StoreParams& p, unsigned* err, int grid,
                              cudaStream_t s, const CUtensorMap* tb2) {
  if (!a_mn && !b_mn)
    return launch_gemm_t<EpiStore, false, false>(ta, tb, g, p, err, grid, s,
                                                 tb2);
  if (!a_mn && b_mn)
    return launch_gemm_t<EpiStore, false, true>(ta, tb, g, p, err, grid, s,
                                                tb2);
  if (a_mn && !b_mn)
    return launch_gemm_t<EpiStore, true, false>(ta, tb, g, p, err, grid, s,
                                                tb2);
  return launch_gemm_t<EpiStore, true, true>(ta, tb, g, p, err, grid, s, tb2);
}

cudaError_t pair_max_active_clusters(int* n) {
  auto kern = k_gemm_pair<EpiStore, false, false>;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM2_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = GEMM2_SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(n, kern, &cfg);
}

cudaError_t launch_gemm_pair_store(bool a_mn, bool b_mn, const CUtensorMap& ta,
                                   const CUtensorMap& tb, const GemmGeom& g,
                                   const StoreParams& p, unsigned* err,
                                   int grid, cudaStream_t s,
                                   const CUtensorMap* tb2) {
  if (!a_mn && !b_mn)
    return launch_gemm_pair_t<EpiStore, false, false>(ta, tb, g, p, err, grid,
                                                      s, tb2);
  if (!a_mn && b_mn)
    return launch_gemm_pair_t<EpiStore, false, true>(ta, tb, g, p, err, grid,
                                                     s, tb2);
  if (a_mn && !b_mn)
    return launch_gemm_pair_t<EpiStore, true, false>(ta, tb, g, p, err, grid,
                                                     s, tb2);
  return launch_gemm_pair_t<EpiStore, true, true>(ta, tb, g, p, err, grid, s,
                                                  tb2);
}

}  // namespace lce
