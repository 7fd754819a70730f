"""Fused linear cross-entropy (the chunked LM-head loss) for NVIDIA GB300.

loss = mean over valid rows of the cross entropy of logits = h W^T against
integer labels, forward and backward, without ever holding the L x V logits
("Training Beyond 1M Tokens", sections "The loss is the first thing to
break" and "The massive logits matrix: chunk it"). The arithmetic runs in
hand-written sm_103a kernels (tcgen05 tensor cores, TMA) behind the C ABI in
include/lce.h; this package is the thin Python binding.

    import chunked_lm_head_gemm_gb300 as lce
    loss = lce.linear_cross_entropy(h, W, labels)       # autograd-aware
    loss, lse = lce.forward(h, W, labels)
    dH, dW = lce.backward(h, W, labels, lse, dloss)
    loss, lse, dH, dW = lce.forward_backward(h, W, labels)  # no recompute
    y = lce.mlp_forward(x, Wg, Wu, Wd)          # sequence-tiled gated MLP
    dx, dWg, dWu, dWd = lce.mlp_backward(x, Wg, Wu, Wd, dy)
    y = lce.sequence_tiled_mlp(x, Wg, Wu, Wd)   # the same, autograd-aware
    from chunked_lm_head_gemm_gb300 import sharded   # rows split over ranks
    loss, lse, dH, dW = sharded.forward_backward(h, W, labels, group)
    from chunked_lm_head_gemm_gb300 import vocab_parallel as vp  # head split
    loss, lse = vp.forward(h, W[v0:v0 + Vs], labels, v0, V, group)
    dH, dW_slice = vp.backward(h, W[v0:v0 + Vs], labels, lse, dloss, v0, V,
                               group)
"""
from ._binding import (IGNORE_INDEX, LCEError, LinearCrossEntropy,
                       SequenceTiledMLP, alloc_workspace, backward, count_valid,
                       default_chunk_rows, forward, forward_backward,
                       get_error, library_path, linear_cross_entropy, load,
                       mlp_backward, mlp_forward, mlp_workspace_size,
                       profile_start, profile_stop, scale_gradients,
                       sequence_tiled_mlp, workspace_size)

__all__ = ["IGNORE_INDEX", "LCEError", "LinearCrossEntropy", "SequenceTiledMLP",
           "alloc_workspace",
           "backward", "count_valid", "default_chunk_rows", "forward",
           "forward_backward", "get_error", "library_path",
           "linear_cross_entropy", "load", "mlp_backward", "mlp_forward",
           "mlp_workspace_size", "profile_start", "profile_stop",
           "scale_gradients", "sequence_tiled_mlp", "workspace_size"]
