"""The loss of a sequence whose rows are split over the processes of a group.

Context parallelism gives each GPU one slice of a long sequence ("Training
Beyond 1M Tokens", section "One GPU is not enough: split the sequence across
many"); the LM-head loss then runs on each slice's rows. The loss of the
whole sequence is the mean over ALL its valid rows, so the shards' own means
cannot simply be averaged: with S_r the sum of the loss terms of shard r and
N_r its valid rows (TRL PR #6845, "TRL: document 1M-token training and add a
context-parallelism example", table "Assumptions", names an evaluation loss
that comes out scaled by the number of shards when this is missed),

    loss  = sum_r S_r / N,        N = sum_r N_r, S_r = N_r loss_r
    dH_r  = (dloss N_r / N) dH'_r             stays on its shard
    dW    = sum_r (dloss N_r / N) dW'_r

where loss_r, dH'_r, dW'_r are the shard's own mean loss and its gradients.
The exchange is one all-reduce of two float64 scalars and one sum of the
V x H fp32 weight gradient. Every loss and gradient value, and the
weighting above, comes from the library's kernels (lce_shard_sums,
lce_combine_shards, lce_scale_gradients); this module only moves data
between the processes of the group. With no group (or a group of one) it
reduces to the single-process call.
"""
from __future__ import annotations

import torch

from . import _binding as B


def _world(group) -> int:
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return 1
    return dist.get_world_size(group)


def exchange(sums: torch.Tensor, group=None) -> torch.Tensor:
    """The shards' (N_r loss_r, N_r) pairs summed in place over `group` (one
    all-reduce of two float64 values); nothing to do without a group."""
    if _world(group) > 1:
        import torch.distributed as dist
        dist.all_reduce(sums, op=dist.ReduceOp.SUM, group=group)
    return sums


def combine_loss(loss_local: torch.Tensor, n_local: torch.Tensor,
                 group=None, dloss: torch.Tensor | None = None):
    """(loss, weight) of the whole sequence from one shard's mean loss and
    valid-row count: loss = sum_r N_r loss_r / sum_r N_r and weight =
    dloss N_r / sum_r N_r (dloss defaults to 1), both 0 when no row of any
    shard is valid. The arithmetic runs in the library; the exchange is one
    all-reduce of two float64 scalars over `group`; no host sync."""
    sums = exchange(B.shard_sums(loss_local, n_local), group)
    return B.combine_shards(sums, n_local, dloss)


def sum_weight_grad(dW: torch.Tensor, group=None) -> torch.Tensor:
    """dW summed in place over the group (fp32, fixed by the backend's
    reduction order)."""
    if _world(group) > 1:
        import torch.distributed as dist
        dist.all_reduce(dW, op=dist.ReduceOp.SUM, group=group)
    return dW


def forward_backward(h: torch.Tensor, W: torch.Tensor, labels: torch.Tensor,
                     group=None, dloss: torch.Tensor | None = None,
                     ignore_index: int = B.IGNORE_INDEX, chunk_rows: int = 0,
                     workspace=None, label_smoothing: float = 0.0,
                     z_loss: float = 0.0):
    """This shard's rows of one sequence: returns (loss, lse, dH, dW) where
    loss is the whole sequence's mean loss (identical on every process), lse
    and dH are this shard's rows, and dW is the weight gradient of the whole
    sequence (summed over the group). dloss defaults to 1. A loss variant
    (label_smoothing, z_loss; the same on every process) is still a mean of
    per-row terms over the valid rows, so it combines the same way."""
    V = W.shape[0]
    loss_r, lse, dH, dW = B.forward_backward(h, W, labels,
                                             ignore_index=ignore_index,
                                             chunk_rows=chunk_rows,
                                             workspace=workspace,
                                             label_smoothing=label_smoothing,
                                             z_loss=z_loss)
    n_r = B.count_valid(labels, V, ignore_index)
    loss, weight = combine_loss(loss_r, n_r, group, dloss)
    B.scale_gradients(dH, dW, weight)
    sum_weight_grad(dW, group)
    return loss, lse, dH, dW
