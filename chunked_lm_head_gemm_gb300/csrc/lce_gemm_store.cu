// Tensor-core contractions with a plain scaled store: dH = (dloss/N) G W and
// dW (+)= (dloss/N) G^T h of the backward, and the building-block GEMM the
// tests use to check every operand layout.
#include "lce_device.cuh"

namespace lce {

cudaError_t launch_gemm_store(bool a_mn, bool b_mn, const CUtensorMap& ta,
                              const CUtensorMap& tb, const GemmGeom& g,
                              const StoreParams& p, unsigned* err, int grid,
                              cudaStream_t s) {
  if (!a_mn && !b_mn)
    return launch_gemm_t<EpiStore, false, false>(ta, tb, g, p, err, grid, s);
  if (!a_mn && b_mn)
    return launch_gemm_t<EpiStore, false, true>(ta, tb, g, p, err, grid, s);
  if (a_mn && !b_mn)
    return launch_gemm_t<EpiStore, true, false>(ta, tb, g, p, err, grid, s);
  return launch_gemm_t<EpiStore, true, true>(ta, tb, g, p, err, grid, s);
}

}  // namespace lce
