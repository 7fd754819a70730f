"""The seeded synthetic inputs follow the recipe they state: deterministic
per seed, the stated shapes and dtypes, exact ignore counts, the Zipf label
law for the 4B workload, and the scaled stress rows of the 32B workload."""
import math

import torch

from chunked_lm_head_gemm_gb300.inputs import (IGNORE_INDEX, MLP_WORKLOADS,
                                               WORKLOADS, Workload,
                                               make_hidden, make_inputs,
                                               make_labels, make_mlp_inputs)


def test_same_seed_same_values_other_seed_other_values():
    a = make_inputs("tiny", seed=0)
    b = make_inputs("tiny", seed=0)
    c = make_inputs("tiny", seed=1)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert not torch.equal(a[0], c[0]) and not torch.equal(a[1], c[1])


def test_tiny_shapes_dtypes_and_ignore_count():
    wl = WORKLOADS["tiny"]
    h, W, y = make_inputs(wl, seed=0)
    assert h.shape == (512, 256) and W.shape == (4096, 256)
    assert h.dtype == torch.float32 and W.dtype == torch.float32
    assert y.dtype == torch.int64 and y.shape == (512,)
    assert int((y == IGNORE_INDEX).sum()) == round(0.10 * 512)
    valid = y[y != IGNORE_INDEX]
    assert int(valid.min()) >= 0 and int(valid.max()) < 4096
    # N(0, 1) hidden, N(0, 0.02^2) weights
    assert abs(h.std().item() - 1.0) < 0.02
    assert abs(W.std().item() - 0.02) < 0.001


def test_ignore_counts_of_every_head_shape():
    for name, wl in WORKLOADS.items():
        y = make_labels(wl, seed=0)
        n_ign = int((y == IGNORE_INDEX).sum())
        want = round(wl.ignore_frac * wl.L)
        if wl.ignore_last:
            assert y[-1].item() == IGNORE_INDEX
            want = max(want, 1)
        assert n_ign == want, name


def test_zipf_labels_follow_the_law():
    """p(id k-1) = k^-s / sum_j j^-s over the 163840 labels of the 4B
    workload: the first ids' frequencies within 4 standard errors."""
    wl = WORKLOADS["qwen3-4b"]
    y = make_labels(wl, seed=0)
    y = y[y != IGNORE_INDEX]
    n = y.numel()
    z = sum(k ** -wl.zipf_s for k in range(1, wl.V + 1))
    counts = torch.bincount(y, minlength=wl.V)
    for k in (1, 2, 3, 10, 100):
        p = k ** -wl.zipf_s / z
        se = math.sqrt(p * (1 - p) / n)
        assert abs(counts[k - 1].item() / n - p) < 4 * se, k
    # rank order holds at the head of the distribution
    assert counts[0] > counts[1] > counts[2] > counts[9]


def test_stress_rows_of_the_32b_workload():
    """1% of rows scaled by 20: on a 2000-row slice exactly 20 rows have a
    norm near 20 * sqrt(H), the rest near sqrt(H)."""
    wl = WORKLOADS["qwen3-32b"].with_rows(2000)
    h = make_hidden(wl, seed=0).float()
    norms = h.norm(dim=1) / math.sqrt(wl.H)
    big = norms > 5.0
    assert int(big.sum()) == 20
    assert torch.all((norms[big] > 18.0) & (norms[big] < 22.0))
    assert torch.all((norms[~big] > 0.9) & (norms[~big] < 1.1))
    assert h.dtype == torch.float32  # widened here for the check
    assert make_hidden(wl, seed=0).dtype == torch.bfloat16


def test_8b_workload_ignores_only_its_last_row():
    y = make_labels(WORKLOADS["qwen3-8b"], seed=0)
    assert int((y == IGNORE_INDEX).sum()) == 1 and y[-1] == IGNORE_INDEX


def test_with_rows_keeps_the_distributions():
    wl = Workload("w", 1000, 64, 500, "bf16", 0.5, 0.02, "uniform",
                  ignore_frac=0.2)
    small = wl.with_rows(300)
    assert small.L == 300 and small.H == 64 and small.V == 500
    assert small.ignore_frac == 0.2 and small.h_scale == 0.5
    y = make_labels(small, seed=2)
    assert int((y == IGNORE_INDEX).sum()) == 60


def test_mlp_inputs_shapes_and_seeds():
    wl = MLP_WORKLOADS["qwen3-0.6b-mlp"].with_rows(64)
    x, Wg, Wu, Wd, dy = make_mlp_inputs(wl, seed=0)
    assert x.shape == (64, 1024) and dy.shape == (64, 1024)
    assert Wg.shape == (3072, 1024) and Wu.shape == (3072, 1024)
    assert Wd.shape == (1024, 3072)
    for t in (x, Wg, Wu, Wd, dy):
        assert t.dtype == torch.bfloat16
    # the five tensors come from five generators
    assert not torch.equal(Wg, Wu)
    again = make_mlp_inputs(wl, seed=0)
    assert all(torch.equal(a, b) for a, b in zip((x, Wg, Wu, Wd, dy), again))
