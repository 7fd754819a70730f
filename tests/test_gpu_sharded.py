"""Row-sharded loss on the GPU, the shards run one after another on one
device: each shard's lce_forward_backward and lce_count_valid, its
(N_r loss_r, N_r) from lce_shard_sums, the pairs summed (standing in for
the all-reduce) and weighed by lce_combine_shards, must give the whole
sequence's loss and gradients ("Training Beyond 1M Tokens", section "One
GPU is not enough: split the sequence across many"). Also the valid-row
count against the oracle, bit for bit, and the combine's edge cases."""
import pytest
import torch

import oracle
import chunked_lm_head_gemm_gb300 as lce
from chunked_lm_head_gemm_gb300 import _binding as B
from chunked_lm_head_gemm_gb300 import sharded
from chunked_lm_head_gemm_gb300.inputs import Workload, make_inputs
from tests.gpu_util import (GRAD_RFRO, LOSS_RTOL, PAIRS, cta_pair, rel_fro,
                            require_gpu, to64)

pytestmark = pytest.mark.gpu

WL = Workload("shards", 1024, 256, 4096, "bf16", 1.0, 0.05, "uniform",
              ignore_frac=0.2)
# ragged shard boundaries (not multiples of the 128-row tile)
BOUNDS = [0, 300, 800, 1024]


@pytest.mark.parametrize("case", ["mixed", "ignored_head"])
def test_count_valid_matches_oracle(case):
    dev = require_gpu()
    _, _, y = make_inputs(WL, seed=3, device=dev)
    if case == "ignored_head":
        y[:500] = -100
    n = B.count_valid(y, WL.V)
    ref, bad = oracle.count_valid(y.cpu(), WL.V)
    assert B.get_error() == 0 and not bad
    assert int(n.item()) == ref
    # an empty label vector counts zero
    empty = torch.empty(0, dtype=torch.int64, device=dev)
    assert int(B.count_valid(empty, WL.V).item()) == 0


def test_count_valid_label_out_of_range():
    dev = require_gpu()
    y = torch.tensor([0, 5, -100, 7, 99, -3], dtype=torch.int64, device=dev)
    n = B.count_valid(y, 8)
    assert B.get_error() == B.LCE_ERR_LABEL_RANGE
    assert int(n.item()) == 3          # 0, 5, 7; 99 and -3 are out of range
    assert oracle.count_valid(y.cpu(), 8) == (3, True)
    assert B.get_error() == 0          # the error word was cleared


@pytest.mark.parametrize("pair", PAIRS, ids=lambda v: "pair" if v else "cta")
def test_sequential_shards_equal_whole_sequence(pair):
    dev = require_gpu()
    h, W, y = make_inputs(WL, seed=5, device=dev)
    dloss = 0.5
    with cta_pair(pair):
        parts = []
        for r0, r1 in zip(BOUNDS[:-1], BOUNDS[1:]):
            loss_r, lse_r, dH_r, dW_r = lce.forward_backward(
                h[r0:r1].contiguous(), W, y[r0:r1].contiguous())
            n_r = B.count_valid(y[r0:r1].contiguous(), WL.V)
            parts.append((loss_r, lse_r, dH_r, dW_r, n_r))
        # the library's combine: each shard's (N_r loss_r, N_r), their sum
        # (the all-reduce of a process group), loss and weight per shard
        total = sum(B.shard_sums(p[0], p[4]) for p in parts)
        d = torch.full((), dloss, device=dev)
        dW = torch.zeros(WL.V, WL.H, dtype=torch.float32, device=dev)
        dH = []
        losses = []
        for loss_r, lse_r, dH_r, dW_r, n_r in parts:
            loss, weight = B.combine_shards(total, n_r, d)
            losses.append(loss)
            lce.scale_gradients(dH_r, dW_r, weight)
            dH.append(dH_r)
            dW += dW_r
        assert all(torch.equal(x, losses[0]) for x in losses)
        dH = torch.cat(dH)
        lse = torch.cat([p[1] for p in parts])
        assert lce.get_error() == 0

        whole = lce.forward_backward(h, W, y)
        lce.scale_gradients(whole[2], whole[3],
                            torch.full((), dloss, device=dev))
    # GPU shards vs GPU whole: same kernels, other tiling and one more bf16
    # rounding of dH after the weight
    assert abs(loss.item() - whole[0].item()) <= 1e-5 * abs(whole[0].item())
    # rows are independent; only the vocabulary split of the sum may differ
    assert torch.max(torch.abs(lse - whole[1])).item() <= 1e-5
    assert rel_fro(to64(dH), to64(whole[2])) <= 4e-3
    assert rel_fro(to64(dW), to64(whole[3])) <= 1e-3

    # and against the float64 oracle on the whole sequence
    hc, Wc, yc = h.cpu(), W.cpu(), y.cpu()
    f = oracle.forward(hc, Wc, yc)
    b = oracle.backward(hc, Wc, yc, dloss=dloss)
    assert abs(loss.item() - f["loss"]) <= LOSS_RTOL * abs(f["loss"])
    assert rel_fro(to64(dH), b["dH"]) <= GRAD_RFRO
    assert rel_fro(to64(dW), b["dW"]) <= GRAD_RFRO


def test_sharded_call_without_group_is_the_single_call():
    dev = require_gpu()
    h, W, y = make_inputs(WL, seed=6, device=dev)
    d = torch.full((), 0.25, device=dev)
    loss, lse, dH, dW = sharded.forward_backward(h, W, y, dloss=d)
    ref = lce.forward_backward(h, W, y)
    lce.scale_gradients(ref[2], ref[3], d)
    assert lce.get_error() == 0
    assert torch.equal(loss, ref[0]) and torch.equal(lse, ref[1])
    assert torch.equal(dH, ref[2]) and torch.equal(dW, ref[3])


def test_combine_shards_edge_cases():
    """N = 0 over all shards gives loss 0 and weight 0; a shard without a
    valid row gets weight 0; a missing dloss counts as 1; the weights of
    the shards sum to dloss."""
    dev = require_gpu()
    n = [torch.tensor([k], dtype=torch.int64, device=dev) for k in (38, 0,
                                                                    24)]
    ls = [torch.tensor(v, dtype=torch.float32, device=dev)
          for v in (2.0, 0.0, 3.5)]
    total = sum(B.shard_sums(l, k) for l, k in zip(ls, n))
    assert total[1].item() == 62.0
    assert total[0].item() == 38 * 2.0 + 24 * 3.5
    d = torch.full((), 0.5, device=dev)
    out = [B.combine_shards(total, k, d) for k in n]
    assert out[0][0].item() == pytest.approx((76.0 + 84.0) / 62.0, rel=1e-7)
    assert out[1][1].item() == 0.0
    assert sum(w.item() for _, w in out) == pytest.approx(0.5, rel=1e-6)
    assert B.combine_shards(total, n[2])[1].item() == pytest.approx(
        24 / 62, rel=1e-7)
    zero = B.shard_sums(ls[1], n[1])
    loss, weight = B.combine_shards(zero, n[1], d)
    assert loss.item() == 0.0 and weight.item() == 0.0
    assert B.get_error() == 0


@pytest.mark.parametrize("eps,zc", [(0.1, 0.0), (0.2, 1e-3)],
                         ids=["eps0.1", "eps0.2-z0.001"])
def test_sequential_shards_with_loss_variant(eps, zc):
    """A loss variant's shards combine as the plain loss's do (the variant
    is still a mean of per-row terms over the valid rows): the shards'
    combined loss and gradients against the oracle's variant on the whole
    sequence."""
    dev = require_gpu()
    h, W, y = make_inputs(WL, seed=7, device=dev)
    var = dict(label_smoothing=eps, z_loss=zc)
    parts = []
    for r0, r1 in zip(BOUNDS[:-1], BOUNDS[1:]):
        loss_r, lse_r, dH_r, dW_r = lce.forward_backward(
            h[r0:r1].contiguous(), W, y[r0:r1].contiguous(), **var)
        parts.append((loss_r, dH_r, dW_r,
                      B.count_valid(y[r0:r1].contiguous(), WL.V)))
    total = sum(B.shard_sums(p[0], p[3]) for p in parts)
    d = torch.full((), 0.75, device=dev)
    dW = torch.zeros(WL.V, WL.H, dtype=torch.float32, device=dev)
    dH = []
    for loss_r, dH_r, dW_r, n_r in parts:
        loss, weight = B.combine_shards(total, n_r, d)
        lce.scale_gradients(dH_r, dW_r, weight)
        dH.append(dH_r)
        dW += dW_r
    assert lce.get_error() == 0
    fb = oracle.forward_backward(h.cpu(), W.cpu(), y.cpu(), dloss=0.75,
                                 **var)
    assert abs(loss.item() - fb["loss"]) <= LOSS_RTOL * abs(fb["loss"])
    assert rel_fro(to64(torch.cat(dH)), fb["dH"]) <= GRAD_RFRO
    assert rel_fro(to64(dW), fb["dW"]) <= GRAD_RFRO
    # the module's call without a group is the single variant call
    s = sharded.forward_backward(h, W, y, dloss=d, **var)
    ref = lce.forward_backward(h, W, y, **var)
    lce.scale_gradients(ref[2], ref[3], d)
    assert torch.equal(s[0], ref[0]) and torch.equal(s[2], ref[2])
    assert torch.equal(s[3], ref[3])
