// Tensor-core contractions whose epilogues carry the loss arithmetic:
//  - forward logits h W^T -> per-row online log-sum-exp partials and the
//    logit at the label ("Training Beyond 1M Tokens", section "The loss is
//    the first thing to break": logits L x V, cross entropy against labels);
//  - backward recompute of the same logits for one row chunk -> bf16
//    softmax - onehot (the gradient of that cross entropy w.r.t. the logits);
//  - the fused forward+backward's logits of one row chunk -> the forward's
//    statistics plus bf16 exponentials relative to each tile's maximum.
#include "lce_device.cuh"

namespace lce {

cudaError_t launch_gemm_lse(const CUtensorMap& ta, const CUtensorMap& tb,
                            const GemmGeom& g, const LseParams& p,
                            unsigned* err, int grid, cudaStream_t s) {
  return launch_gemm_t<EpiLse, false, false>(ta, tb, g, p, err, grid, s);
}

// tg: store map of the chunk's gradient logits (tmap_store_box), handed to
// the kernel in the second-B slot, which this contraction does not use.
cudaError_t launch_gemm_grad(const CUtensorMap& ta, const CUtensorMap& tb,
                             const CUtensorMap& tg, const GemmGeom& g,
                             const GradParams& p, unsigned* err, int grid,
                             cudaStream_t s) {
  return launch_gemm_t<EpiGrad, false, false>(ta, tb, g, p, err, grid, s,
                                              &tg);
}

// te: store map of the chunk's exponentials (tmap_store_box), handed to the
// kernel in the second-B slot, which this contraction does not use.
cudaError_t launch_gemm_fused(const CUtensorMap& ta, const CUtensorMap& tb,
                              const CUtensorMap& te, const GemmGeom& g,
                              const FusedParams& p, unsigned* err, int grid,
                              cudaStream_t s) {
  return launch_gemm_t<EpiFused, false, false>(ta, tb, g, p, err, grid, s,
                                               &te);
}

cudaError_t launch_gemm_pair_lse(const CUtensorMap& ta, const CUtensorMap& tb,
                                 const GemmGeom& g, const LseParams& p,
                                 unsigned* err, int grid, cudaStream_t s) {
  return launch_gemm_pair_t<EpiLse, false, false>(ta, tb, g, p, err, grid, s);
}

cudaError_t launch_gemm_pair_grad(const CUtensorMap& ta, const CUtensorMap& tb,
                                  const CUtensorMap& tg, const GemmGeom& g,
                                  const GradParams& p, unsigned* err, int grid,
                                  cudaStream_t s) {
  return launch_gemm_pair_t<EpiGrad, false, false>(ta, tb, g, p, err, grid, s,
                                                   &tg);
}

cudaError_t launch_gemm_pair_fused(const CUtensorMap& ta,
                                   const CUtensorMap& tb,
                                   const CUtensorMap& te, const GemmGeom& g,
                                   const FusedParams& p, unsigned* err,
                                   int grid, cudaStream_t s) {
  return launch_gemm_pair_t<EpiFused, false, false>(ta, tb, g, p, err, grid,
                                                    s, &te);
}

}  // namespace lce
