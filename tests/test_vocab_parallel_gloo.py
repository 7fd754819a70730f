"""Vocabulary-parallel exchange on CPU: two gloo processes each hold a slice
of the head and produce their slice's per-row statistics with the float64
oracle (standing in for the GPU library); chunked_lm_head_gemm_gb300.
vocab_parallel gathers them in rank order and sums the dH partials. Merging
the gathered statistics by the log-sum-exp identity must give the oracle's
lse and loss on the whole vocabulary."""
import os
import socket

import numpy as np
import pytest
import torch

L, H, V = 40, 12, 50
SPLIT = 29                 # rank 0 holds ids [0, 29), rank 1 [29, 50)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    g = torch.Generator().manual_seed(3)
    h = torch.randn(L, H, generator=g, dtype=torch.float64)
    W = 0.4 * torch.randn(V, H, generator=g, dtype=torch.float64)
    y = torch.randint(0, V, (L,), generator=g, dtype=torch.int64)
    y[::7] = -100
    return h, W, y


def _rank_main(rank, world, port, out_dir):
    import oracle
    from chunked_lm_head_gemm_gb300 import vocab_parallel as vp
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                            rank=rank, world_size=world)
    try:
        h, W, y = _inputs()
        v0, v1 = (0, SPLIT) if rank == 0 else (SPLIT, V)
        yl = y.clone()
        local = (y >= v0) & (y < v1)
        yl[~local] = -100
        yl[local] -= v0
        f = oracle.forward(h, W[v0:v1], yl, nthreads=1)
        # the slice's statistics as (m, s) = (its lse, 1), and its label
        # logits (0 for labels in the other slice)
        zy = np.where(local.numpy(), f["zy"], 0.0)
        stats = torch.tensor(np.stack([f["lse"], np.ones(L), zy]))
        allst = vp.gather_stats(stats)
        part = torch.full((L, H), float(rank + 1), dtype=torch.float64)
        vp.sum_partials(part)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"),
                 allst=allst.numpy(), part=part.numpy())
    finally:
        dist.destroy_process_group()


def test_two_rank_gather_merges_to_whole_vocabulary(tmp_path, oracle_mod):
    import torch.multiprocessing as mp
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2,
             join=True)
    r = [np.load(tmp_path / f"rank{k}.npz") for k in range(2)]
    np.testing.assert_array_equal(r[0]["allst"], r[1]["allst"])
    allst = r[0]["allst"]                      # [P, 3, L], rank order
    assert allst.shape == (2, 3, L)
    m, s, zy = allst[:, 0], allst[:, 1], allst[:, 2]
    M = m.max(axis=0)
    lse = M + np.log((s * np.exp(m - M)).sum(axis=0))
    h, W, y = _inputs()
    f = oracle_mod.forward(h, W, y, nthreads=1)
    np.testing.assert_allclose(lse, f["lse"], rtol=0, atol=1e-12)
    valid = (y != -100).numpy()
    loss = float(np.mean(lse[valid] - zy.sum(axis=0)[valid]))
    assert abs(loss - f["loss"]) <= 1e-12
    # the dH partials are summed, identical on both ranks
    for k in range(2):
        assert np.all(r[k]["part"] == 3.0)


EPS, ZC = 0.1, 1e-2


def _rank_main_smoothed(rank, world, port, out_dir):
    import oracle
    from chunked_lm_head_gemm_gb300 import vocab_parallel as vp
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                            rank=rank, world_size=world)
    try:
        h, W, y = _inputs()
        v0, v1 = (0, SPLIT) if rank == 0 else (SPLIT, V)
        yl = y.clone()
        local = (y >= v0) & (y < v1)
        yl[~local] = -100
        yl[local] -= v0
        f = oracle.forward(h, W[v0:v1], yl, nthreads=1)
        zy = np.where(local.numpy(), f["zy"], 0.0)
        # the fourth row under label smoothing: the slice's logit sums
        zsum = (h @ W[v0:v1].T).sum(dim=1).numpy()
        stats = torch.tensor(np.stack([f["lse"], np.ones(L), zy, zsum]))
        allst = vp.gather_stats(stats)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"),
                 allst=allst.numpy())
    finally:
        dist.destroy_process_group()


def test_two_rank_gather_of_smoothed_statistics(tmp_path, oracle_mod):
    """Four rows per slice under label smoothing: gathered in rank order,
    merged per row they give the oracle's smoothed loss with z-loss over
    the whole vocabulary."""
    import torch.multiprocessing as mp
    mp.spawn(_rank_main_smoothed, args=(2, _free_port(), str(tmp_path)),
             nprocs=2, join=True)
    r = [np.load(tmp_path / f"rank{k}.npz") for k in range(2)]
    np.testing.assert_array_equal(r[0]["allst"], r[1]["allst"])
    allst = r[0]["allst"]
    assert allst.shape == (2, 4, L)
    m, s, zy, zs = allst[:, 0], allst[:, 1], allst[:, 2], allst[:, 3]
    M = m.max(axis=0)
    lse = M + np.log((s * np.exp(m - M)).sum(axis=0))
    h, W, y = _inputs()
    f = oracle_mod.forward(h, W, y, nthreads=1, label_smoothing=EPS,
                           z_loss=ZC)
    valid = (y != -100).numpy()
    term = (lse - (1 - EPS) * zy.sum(axis=0) - EPS / V * zs.sum(axis=0)
            + ZC * lse ** 2)
    assert abs(float(np.mean(term[valid])) - f["loss"]) <= 1e-12
