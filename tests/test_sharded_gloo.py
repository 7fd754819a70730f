"""Row-sharded loss on CPU: two gloo processes each hold a slice of one
sequence's rows, compute their shard's mean loss and gradients with the
float64 oracle (standing in for the GPU library, which needs a device),
exchange their (N_r loss_r, N_r) pairs and weight gradients with
chunked_lm_head_gemm_gb300.sharded, and weigh them as the library's
lce_combine_shards does (that kernel itself is tested on the GPU). The
result must equal the oracle on the whole sequence: the loss as the mean
over ALL valid rows (not the mean of the shards' means), each shard's dH
rows, and the summed dW ("Training Beyond 1M Tokens", section "One GPU is
not enough: split the sequence across many")."""
import os
import socket

import numpy as np
import pytest
import torch

L, H, V = 72, 16, 40
SPLIT = 48                # rank 0 holds rows [0, 48), rank 1 rows [48, 72)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(case: str):
    g = torch.Generator().manual_seed(7)
    h = torch.randn(L, H, generator=g, dtype=torch.float64)
    W = 0.3 * torch.randn(V, H, generator=g, dtype=torch.float64)
    y = torch.randint(0, V, (L,), generator=g, dtype=torch.int64)
    if case == "uneven":
        y[:10] = -100             # shard 0: 38 valid rows, shard 1: 24
    elif case == "shard_empty":
        y[SPLIT:] = -100          # shard 1 has no valid row
    elif case == "all_ignored":
        y[:] = -100
    return h, W, y


def _rank_main(rank, world, port, case, out_dir):
    import oracle
    from chunked_lm_head_gemm_gb300 import sharded
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                            rank=rank, world_size=world)
    try:
        h, W, y = _inputs(case)
        rows = slice(0, SPLIT) if rank == 0 else slice(SPLIT, L)
        hs, ys = h[rows], y[rows]
        fw = oracle.forward(hs, W, ys, nthreads=2)
        bw = oracle.backward(hs, W, ys, dloss=1.0, nthreads=2)
        # the shard's loss travels as fp32, as the library returns it
        loss_r = float(np.float32(fw["loss"]))
        n_r = fw["n_valid"]
        sums = sharded.exchange(torch.tensor([n_r * loss_r, float(n_r)],
                                             dtype=torch.float64))
        total = sums[1].item()
        loss = sums[0].item() / total if total > 0 else 0.0
        weight = n_r / total if total > 0 else 0.0
        dloss = 0.75
        dH = torch.from_numpy(bw["dH"]) * (weight * dloss)
        dW = torch.from_numpy(bw["dW"]) * (weight * dloss)
        sharded.sum_weight_grad(dW)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), loss=loss,
                 loss_r=fw["loss"], weight=weight, dH=dH.numpy(),
                 dW=dW.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", ["uneven", "shard_empty", "all_ignored"])
def test_two_rank_gloo_matches_whole_sequence(case, tmp_path, oracle_mod):
    import torch.multiprocessing as mp
    mp.spawn(_rank_main, args=(2, _free_port(), case, str(tmp_path)),
             nprocs=2, join=True)
    r = [np.load(tmp_path / f"rank{k}.npz") for k in range(2)]

    h, W, y = _inputs(case)
    whole_f = oracle_mod.forward(h, W, y, nthreads=2)
    whole_b = oracle_mod.backward(h, W, y, dloss=0.75, nthreads=2)
    n = whole_f["n_valid"]

    for k in range(2):
        # the loss travels as fp32 from each shard; the combine is float64
        assert abs(float(r[k]["loss"]) - whole_f["loss"]) <= \
            1e-6 * max(1.0, abs(whole_f["loss"]))
    np.testing.assert_allclose(np.concatenate([r[0]["dH"], r[1]["dH"]]),
                               whole_b["dH"], rtol=1e-6, atol=1e-12)
    for k in range(2):
        np.testing.assert_allclose(r[k]["dW"], whole_b["dW"], rtol=1e-6,
                                   atol=1e-12)
    if case == "uneven":
        # the pitfall the combine avoids: averaging the shards' own means
        naive = 0.5 * (float(r[0]["loss_r"]) + float(r[1]["loss_r"]))
        assert abs(naive - whole_f["loss"]) > 1e-3
        assert abs(float(r[0]["weight"]) - 38 / 62) < 1e-12
    if case == "shard_empty":
        assert float(r[1]["weight"]) == 0.0 and float(r[0]["weight"]) == 1.0
    if case == "all_ignored":
        assert n == 0 and float(r[0]["loss"]) == 0.0
        assert not np.any(r[0]["dW"]) and not np.any(r[1]["dH"])


def test_single_process_exchange_is_identity():
    from chunked_lm_head_gemm_gb300 import sharded
    sums = torch.tensor([42.5, 17.0], dtype=torch.float64)
    assert torch.equal(sharded.exchange(sums.clone()), sums)
    dW = torch.randn(3, 4)
    assert torch.equal(sharded.sum_weight_grad(dW.clone()), dW)
