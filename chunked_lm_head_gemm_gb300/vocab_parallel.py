"""The loss with the LM head split by vocabulary over the processes of a group.

Each process holds all of h and one slice of the head's rows, W[v0, v0 + Vs)
of a vocabulary of V_total (tensor parallelism on the head). "Training Beyond
1M Tokens", section "The massive logits matrix: chunk it", explains that rows
split cleanly because the softmax runs along one row's vocabulary; split the
vocabulary instead and each row's log-sum-exp must be merged from the slices:

    forward   each slice: m_r = max_j z_ij, s_r = sum_j exp(z_ij - m_r), and
              the label logit if the label is in the slice (else 0)
              exchange: all-gather of (m, s, zy), 3 L floats per process
              every process: lse = M + ln sum_r s_r exp(m_r - M), M = max_r m_r,
              loss = mean over valid rows of lse - z_y (same bits everywhere)
    backward  each slice: G_r = dloss/N (exp(z - lse) - [j == y]) on its
              columns, dW_r = G_r^T h (stays local), dH_r = G_r W_r
              exchange: all-reduce (sum) of the fp32 dH_r, L H floats

With label smoothing each slice also gives its per-row sum of logits (a
fourth gathered row), and the merged loss and the slices' G are the
smoothed cross entropy's; a z-loss needs nothing more than the merged lse.

Every loss and gradient value comes from the library's kernels; this module
only moves the statistics and partial sums between processes. With no group
(or a group of one) the one slice is the whole vocabulary.
"""
from __future__ import annotations

import torch

from . import _binding as B


def _world(group) -> int:
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return 1
    return dist.get_world_size(group)


def gather_stats(stats: torch.Tensor, group=None) -> torch.Tensor:
    """stats [R, L] (m, s, zy and, under label smoothing, zsum of this
    process's slice) -> [P, R, L] in rank order, the same on every
    process."""
    world = _world(group)
    if world == 1:
        return stats.unsqueeze(0)
    import torch.distributed as dist
    out = torch.empty((world * stats.shape[0],) + tuple(stats.shape[1:]),
                      dtype=stats.dtype, device=stats.device)
    dist.all_gather_into_tensor(out, stats.contiguous(), group=group)
    return out.view((world,) + tuple(stats.shape))


def sum_partials(dH_part: torch.Tensor, group=None) -> torch.Tensor:
    """The slices' dH partials summed in place over the group (fp32)."""
    if _world(group) > 1:
        import torch.distributed as dist
        dist.all_reduce(dH_part, op=dist.ReduceOp.SUM, group=group)
    return dH_part


def _merge(rows, labels, V_total, group, ignore_index, label_smoothing,
           z_loss):
    """This slice's statistics rows -> gathered over the group -> merged
    (loss, lse) of the whole vocabulary."""
    allst = gather_stats(torch.stack(rows), group)
    col = [allst[:, r].contiguous() for r in range(len(rows))]
    return B.combine_slices(col[0], col[1], col[2], labels, V_total,
                            ignore_index,
                            zsum=col[3] if len(col) == 4 else None,
                            label_smoothing=label_smoothing, z_loss=z_loss)


def forward(h: torch.Tensor, W_slice: torch.Tensor, labels: torch.Tensor,
            v0: int, V_total: int, group=None,
            ignore_index: int = B.IGNORE_INDEX, workspace=None,
            label_smoothing: float = 0.0, z_loss: float = 0.0):
    """Returns (loss, lse [L]) of the whole vocabulary on every process."""
    rows = B.forward_slice(h, W_slice, labels, v0, V_total, ignore_index,
                           workspace, label_smoothing=label_smoothing,
                           z_loss=z_loss)
    return _merge(rows, labels, V_total, group, ignore_index,
                  label_smoothing, z_loss)


def backward(h: torch.Tensor, W_slice: torch.Tensor, labels: torch.Tensor,
             lse: torch.Tensor, dloss: torch.Tensor, v0: int, V_total: int,
             group=None, ignore_index: int = B.IGNORE_INDEX,
             chunk_rows: int = 0, workspace=None,
             label_smoothing: float = 0.0, z_loss: float = 0.0,
             compute_dH: bool = True, compute_dW: bool = True):
    """Returns (dH [L,H] float32, summed over the group; dW of this slice
    [Vs,H] float32), None for a gradient not asked for (every process must
    ask for dH alike: its sum is a collective)."""
    dH_part, dW = B.backward_slice(h, W_slice, labels, lse, dloss, v0,
                                   V_total, ignore_index, chunk_rows,
                                   workspace, label_smoothing=label_smoothing,
                                   z_loss=z_loss, compute_dH=compute_dH,
                                   compute_dW=compute_dW)
    if dH_part is not None:
        dH_part = sum_partials(dH_part, group)
    return dH_part, dW


def exp_workspace(h: torch.Tensor, W_slice: torch.Tensor) -> torch.Tensor:
    """Workspace for forward_exp / backward_exp (L x round_up(Vs, 8) bf16
    exponentials and their tile maxima, plus the usual statistics)."""
    return B.slice_exp_workspace(h.shape[0], h.shape[1], W_slice.shape[0],
                                 h.dtype, h.device)


def forward_exp(h: torch.Tensor, W_slice: torch.Tensor, labels: torch.Tensor,
                v0: int, V_total: int, workspace: torch.Tensor, group=None,
                ignore_index: int = B.IGNORE_INDEX,
                label_smoothing: float = 0.0, z_loss: float = 0.0):
    """forward, keeping this slice's exponentials in `workspace` so that
    backward_exp need not recompute the logits."""
    rows = B.forward_slice_exp(h, W_slice, labels, v0, V_total, workspace,
                               ignore_index, label_smoothing=label_smoothing,
                               z_loss=z_loss)
    return _merge(rows, labels, V_total, group, ignore_index,
                  label_smoothing, z_loss)


def backward_exp(h: torch.Tensor, W_slice: torch.Tensor, labels: torch.Tensor,
                 lse: torch.Tensor, dloss: torch.Tensor, v0: int, V_total: int,
                 workspace: torch.Tensor, group=None,
                 ignore_index: int = B.IGNORE_INDEX,
                 label_smoothing: float = 0.0, z_loss: float = 0.0,
                 compute_dH: bool = True, compute_dW: bool = True):
    """backward from the exponentials forward_exp kept (same workspace)."""
    dH_part, dW = B.backward_slice_exp(h, W_slice, labels, lse, dloss, v0,
                                       V_total, workspace, ignore_index,
                                       label_smoothing=label_smoothing,
                                       z_loss=z_loss, compute_dH=compute_dH,
                                       compute_dW=compute_dW)
    if dH_part is not None:
        dH_part = sum_partials(dH_part, group)
    return dH_part, dW


class VocabParallelCrossEntropy(torch.autograd.Function):
    """The loss of the whole vocabulary from this process's head slice, as
    an autograd Function: forward returns the merged loss (the same on every
    process of the group); backward returns dH summed over the group and
    this slice's dW. keep_exp=True keeps the slice's exponentials between
    forward and backward (no recompute, L x Vs x 2 bytes of workspace held
    until backward); else only lse is kept and the backward recomputes.
    label_smoothing / z_loss select the loss variant (the same on every
    process)."""

    @staticmethod
    def forward(ctx, h, W_slice, labels, v0, V_total, group=None,
                ignore_index=B.IGNORE_INDEX, keep_exp=False,
                label_smoothing=0.0, z_loss=0.0):
        ctx.v0, ctx.V_total, ctx.group = v0, V_total, group
        ctx.ignore_index, ctx.keep_exp = ignore_index, keep_exp
        ctx.w_dtype, ctx.h_dtype = W_slice.dtype, h.dtype
        ctx.variant = dict(label_smoothing=label_smoothing, z_loss=z_loss)
        if keep_exp:
            ws = exp_workspace(h, W_slice)
            loss, lse = forward_exp(h, W_slice, labels, v0, V_total, ws,
                                    group, ignore_index, **ctx.variant)
            ctx.ws = ws
        else:
            loss, lse = forward(h, W_slice, labels, v0, V_total, group,
                                ignore_index, **ctx.variant)
            ctx.ws = None
        ctx.save_for_backward(h, W_slice, labels, lse)
        return loss

    @staticmethod
    def backward(ctx, dloss):
        h, W_slice, labels, lse = ctx.saved_tensors
        want = dict(compute_dH=ctx.needs_input_grad[0],
                    compute_dW=ctx.needs_input_grad[1])
        if not any(want.values()):
            ctx.ws = None
            return (None,) * 10
        if ctx.keep_exp:
            dH, dW = backward_exp(h, W_slice, labels, lse, dloss, ctx.v0,
                                  ctx.V_total, ctx.ws, ctx.group,
                                  ctx.ignore_index, **ctx.variant, **want)
            ctx.ws = None
        else:
            dH, dW = backward(h, W_slice, labels, lse, dloss, ctx.v0,
                              ctx.V_total, ctx.group, ctx.ignore_index,
                              **ctx.variant, **want)
        return (dH.to(ctx.h_dtype) if dH is not None else None,
                dW.to(ctx.w_dtype) if dW is not None else None, None, None,
                None, None, None, None, None, None)


def vocab_parallel_cross_entropy(h, W_slice, labels, v0: int, V_total: int,
                                 group=None,
                                 ignore_index: int = B.IGNORE_INDEX,
                                 keep_exp: bool = False,
                                 label_smoothing: float = 0.0,
                                 z_loss: float = 0.0):
    return VocabParallelCrossEntropy.apply(h, W_slice, labels, v0, V_total,
                                           group, ignore_index, keep_exp,
                                           label_smoothing, z_loss)
