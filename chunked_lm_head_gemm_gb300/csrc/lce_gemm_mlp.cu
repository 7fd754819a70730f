// Tensor-core contractions of the sequence-tiled gated MLP ("Training
// Beyond 1M Tokens", section "One GPU is not enough: split the sequence
// across many": one MLP line is down_proj(act_fn(gate_proj(x)) *
// up_proj(x)), act_fn = SiLU): the gate and up projections of a row chunk in
// one contraction whose epilogue forms silu(g) * u, and the backward
// contraction da = dy Wd whose epilogue forms dg and du. The plain
// projections reuse the store contractions.
#include "lce_device.cuh"

namespace lce {

cudaError_t launch_gemm_swiglu(bool pair, const CUtensorMap& ta,
                               const CUtensorMap& tb, const CUtensorMap& tb2,
                               const GemmGeom& g, const SwigluParams& p,
                               unsigned* err, int grid, cudaStream_t s) {
  return pair ? launch_gemm_pair_t<EpiSwiGLU, false, false>(ta, tb, g, p, err,
                                                            grid, s, &tb2)
              : launch_gemm_t<EpiSwiGLU, false, false>(ta, tb, g, p, err,
                                                       grid, s, &tb2);
}

cudaError_t launch_gemm_swiglu_bwd(bool pair, const CUtensorMap& ta,
                                   const CUtensorMap& tb,
                                   const CUtensorMap& tb2, const GemmGeom& g,
                                   const SwigluBwdParams& p, unsigned* err,
                                   int grid, cudaStream_t s) {
  return pair ? launch_gemm_pair_t<EpiSwiGLUBwd, false, true>(
                    ta, tb, g, p, err, grid, s, &tb2)
              : launch_gemm_t<EpiSwiGLUBwd, false, true>(ta, tb, g, p, err,
                                                         grid, s, &tb2);
}

}  // namespace lce
