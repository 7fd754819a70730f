"""Seeded synthetic inputs for the chunked LM-head cross-entropy.

This module holds no arithmetic of the method: it only draws hidden states,
LM-head weights and labels with the shapes and distributions of the
workloads, so that the CUDA path and the float64 oracle can be fed the very
same values. The pages measure on PG-19 text with Qwen3 models; neither is
available, so these draws stand in for them, keeping the Qwen3 head shapes
(hidden size H, vocabulary V = 151936) and the per-GPU sequence lengths.

Recipe (one ``torch.Generator`` per tensor, seeded ``seed * 1000 + k``):
  k=0 hidden h[L,H]:  N(0,1) * h_scale, drawn in fp32, then cast to ``dtype``
  k=1 weights W[V,H]: N(0, w_std^2), drawn in fp32, then cast to ``dtype``
  k=2 labels y[L]:    uniform over [0, V), or Zipf(s) rank k -> id k-1
                      (inverse CDF in float64 on uniform draws)
  k=3 ignore mask:    the first round(p*L) indices of a random permutation
                      are set to ignore_index (so N is exact), or only the
                      last row (shifted-label causal LM)
  k=4 stress rows:    the first round(q*L) indices of a random permutation
                      have their hidden state multiplied by ``stress_scale``
"""
from __future__ import annotations

import dataclasses

import torch

IGNORE_INDEX = -100


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    L: int
    H: int
    V: int
    dtype: str            # "bf16" or "f32": the type h and W are stored in
    h_scale: float = 1.0
    w_std: float = 0.02
    labels: str = "uniform"   # "uniform" or "zipf"
    zipf_s: float = 1.1
    ignore_frac: float = 0.0
    ignore_last: bool = False
    stress_frac: float = 0.0
    stress_scale: float = 1.0

    def with_rows(self, L: int) -> "Workload":
        """The same distributions with another row count (a row slice)."""
        return dataclasses.replace(self, L=L, name=f"{self.name}[L={L}]")


WORKLOADS = {
    # small case: fp32 inputs, 10% ignored
    "tiny": Workload("tiny", 512, 256, 4096, "f32", 1.0, 0.02, "uniform",
                     ignore_frac=0.10),
    # Qwen3-0.6B head shape
    "qwen3-0.6b": Workload("qwen3-0.6b", 32768, 1024, 151936, "bf16", 0.5,
                           0.02, "uniform", ignore_frac=0.05),
    # Qwen3-4B head shape at the 160k single-card length
    "qwen3-4b": Workload("qwen3-4b", 163840, 2560, 151936, "bf16", 1.0, 0.02,
                         "zipf", 1.1, ignore_frac=0.02),
    # Qwen3-8B head shape, one 1M-token sequence's per-GPU shard (1M / 8)
    "qwen3-8b": Workload("qwen3-8b", 131072, 4096, 151936, "bf16", 1.0, 0.015,
                         "uniform", ignore_last=True),
    # Qwen3-32B head shape, 1% of rows scaled x20 (large logits)
    "qwen3-32b": Workload("qwen3-32b", 65536, 5120, 151936, "bf16", 1.0, 0.02,
                          "uniform", ignore_frac=0.10, stress_frac=0.01,
                          stress_scale=20.0),
}


def _gen(seed: int, k: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + k)
    return g


def _tdtype(name: str):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def make_labels(wl: Workload, seed: int = 0) -> torch.Tensor:
    """int64 labels on the CPU (cheap at every size)."""
    g = _gen(seed, 2, "cpu")
    if wl.labels == "uniform":
        y = torch.randint(0, wl.V, (wl.L,), generator=g, dtype=torch.int64)
    elif wl.labels == "zipf":
        ranks = torch.arange(1, wl.V + 1, dtype=torch.float64)
        w = ranks.pow(-wl.zipf_s)
        cdf = torch.cumsum(w, 0)
        cdf = cdf / cdf[-1]
        u = torch.rand(wl.L, generator=g, dtype=torch.float64)
        y = torch.searchsorted(cdf, u).clamp_(max=wl.V - 1).to(torch.int64)
    else:
        raise ValueError(wl.labels)
    if wl.ignore_last:
        y[-1] = IGNORE_INDEX
    n_ign = int(round(wl.ignore_frac * wl.L))
    if n_ign:
        perm = torch.randperm(wl.L, generator=_gen(seed, 3, "cpu"))
        y[perm[:n_ign]] = IGNORE_INDEX
    return y


def make_hidden(wl: Workload, seed: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(seed, 0, device)
    h = torch.randn(wl.L, wl.H, generator=g, device=device,
                    dtype=torch.float32)
    if wl.h_scale != 1.0:
        h.mul_(wl.h_scale)
    n_st = int(round(wl.stress_frac * wl.L))
    if n_st:
        perm = torch.randperm(wl.L, generator=_gen(seed, 4, "cpu"))
        h[perm[:n_st].to(h.device)] *= wl.stress_scale
    return h.to(_tdtype(wl.dtype))


def make_weight(wl: Workload, seed: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(seed, 1, device)
    out = torch.empty(wl.V, wl.H, device=device, dtype=_tdtype(wl.dtype))
    # draw in fp32 slabs of at most 2^26 elements, cast each into place
    rows = max(1, (1 << 26) // max(1, wl.H))
    for r0 in range(0, wl.V, rows):
        r1 = min(wl.V, r0 + rows)
        slab = torch.empty(r1 - r0, wl.H, device=device, dtype=torch.float32)
        slab.normal_(0.0, wl.w_std, generator=g)
        out[r0:r1].copy_(slab)
    return out


def make_inputs(wl: Workload | str, seed: int = 0, device="cpu"):
    """Returns (h[L,H], W[V,H], labels[L] int64), h and W on ``device``."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    y = make_labels(wl, seed)
    h = make_hidden(wl, seed, device)
    W = make_weight(wl, seed, device)
    return h, W, y.to(device)



@dataclasses.dataclass(frozen=True)
class MlpWorkload:
    """A Qwen3 MLP (gate/up I x H, down H x I) over L rows, all bf16."""
    name: str
    L: int
    H: int
    I: int
    x_scale: float = 1.0
    w_std: float = 0.02

    def with_rows(self, L: int) -> "MlpWorkload":
        return dataclasses.replace(self, L=L, name=f"{self.name}[L={L}]")


# Qwen3 MLP widths (hidden H -> intermediate I), one 1M-token sequence's
# per-GPU shard of 131072 rows (1M over 8 GPUs)
MLP_WORKLOADS = {
    "qwen3-0.6b-mlp": MlpWorkload("qwen3-0.6b-mlp", 131072, 1024, 3072),
    "qwen3-4b-mlp": MlpWorkload("qwen3-4b-mlp", 131072, 2560, 9728),
    "qwen3-8b-mlp": MlpWorkload("qwen3-8b-mlp", 131072, 4096, 12288),
    "qwen3-32b-mlp": MlpWorkload("qwen3-32b-mlp", 131072, 5120, 25600),
}


def make_mlp_inputs(wl: MlpWorkload, seed: int = 0, device="cpu"):
    """Returns (x [L,H], Wg [I,H], Wu [I,H], Wd [H,I], dy [L,H]), bf16;
    generators seed*1000 + 10..14."""
    def draw(shape, k, std):
        g = _gen(seed, k, device)
        t = torch.empty(*shape, device=device, dtype=torch.float32)
        t.normal_(0.0, std, generator=g)
        return t.to(torch.bfloat16)
    x = draw((wl.L, wl.H), 10, wl.x_scale)
    Wg = draw((wl.I, wl.H), 11, wl.w_std)
    Wu = draw((wl.I, wl.H), 12, wl.w_std)
    Wd = draw((wl.H, wl.I), 13, wl.w_std)
    dy = draw((wl.L, wl.H), 14, 1.0)
    return x, Wg, Wu, Wd, dy
