#!/usr/bin/env python3
"""Benchmark: fused linear cross-entropy forward + backward on GB300.

One step = the loss and its gradients (dloss = 1) over one synthetic batch
of the chosen head shape (default: the Qwen3-8B head at one 1M-token
sequence's per-GPU shard, L=131072, H=4096, V=151936), inputs resident in
HBM, by one of the library's two paths:
  --mode separate  lce_forward + lce_backward (the backward recomputes the
                   logits chunk by chunk)
  --mode fused     lce_forward_backward + lce_scale_gradients (logits
                   computed once; default)
Both paths are timed; the line reports the --mode one and lists both under
"modes". Prints one JSON line (rank 0):

  value        whole-job tokens/s (rows of h per second), device-timed with
               CUDA events around exactly --steps steps
  roofline     the dominant kernel: algorithmic flops per launch / its
               event-measured launch duration, against the bf16 tensor peak
  cpu_baseline the float64 oracle timed on this host's cores on a bounded
               row sample of the same workload (N=1, rank 0)
  e2e          the same metric with pinned-host inputs copied in and the
               results (loss, dH, dW) copied out inside the timed region
  clocks       nvidia-smi samples taken during the timed region

--impl reference times the float64 oracle instead (host cores, bounded row
sample per step) and prints the same line with "impl": "reference".
--workload mlp times the sequence-tiled gated MLP (lce_mlp_forward +
lce_mlp_backward) on a Qwen3 MLP shape instead (--config qwen3-8b-mlp ...).
--gpus N under torchrun: N independent replicas, one per GPU (the library
has no multi-GPU path), weak scaling, max time over ranks.
Measurement modes that print their own JSON line instead of the benchmark:
--layout-sweep M,N,K (the contraction in its four operand layouts) and
--forward-static (lce_forward_static against lce_forward).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("fused linear-CE fwd+bwd tokens/s and TFLOPS "
          "(fraction of GB300 BF16 peak)")
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "hbm_gbs": 6800.0}
L2_BYTES = 129 * 1024 * 1024


def _flatten(d, out=None):
    out = {} if out is None else out
    if isinstance(d, dict):
        for k, v in d.items():
            if isinstance(v, (int, float)) and not isinstance(v, bool):
                out.setdefault(k, float(v))
            else:
                _flatten(v, out)
    return out


# The pages' whole-step number for the workload that is exactly one GPU's
# shard of their run: Qwen3-8B, one 1M-token sequence over 8 H100s, 131072
# rows per GPU (TRL PR #6845 page, "TRL: document 1M-token training and add
# a context-parallelism example", table under "Measured"). Context only.
PAGES_STEP = {
    "qwen3-8b": {"model": "Qwen3-8B", "tokens": 1048576, "gpus": "8 x H100",
                 "s_per_step": 364.0, "peak_gb": 56.2},
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            flat = _flatten(json.load(open(path)))
            peaks = dict(FALLBACK_PEAKS)
            found = False
            for k in FALLBACK_PEAKS:
                if k in flat:
                    peaks[k] = flat[k]
                    found = True
            if found:
                return peaks, "measured"
        except Exception:  # noqa: BLE001 - fall back on any parse problem
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments and blank space, so that a
    comment edit does not count as a kernel change. String literals with
    comment markers in them are kept as they are (the csrc files have none
    that matter: a changed literal still changes the hash)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_hash() -> str:
    """Hash of the CUDA library's code (comments and spacing ignored)."""
    csrc = os.path.join(ROOT, "chunked_lm_head_gemm_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(f.encode())
            h.update(_code_only(open(os.path.join(csrc, f)).read()).encode())
    return h.hexdigest()[:16]


def load_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if
    it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
    except Exception:  # noqa: BLE001
        return None
    e = d.get(kernel, {}).get(workload)
    if not e or e.get("source_hash") != source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
               "sw_power_cap")

    def __init__(self, device_index: int):
        import torch
        self.proc = None
        self.err = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.target = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception as e:  # noqa: BLE001
            self.target = str(device_index)
            self.err = repr(e)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.target,
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception as e:  # noqa: BLE001
            self.err = repr(e)

    def stop(self) -> dict:
        if self.proc is None:
            return {"error": self.err or "nvidia-smi not started"}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"error": "no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_median": statistics.median(power),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# reference arm and CPU baseline: the float64 oracle on host cores
# ---------------------------------------------------------------------------

def _oracle_rate_macs(h, W, y) -> float:
    """Multiply-adds per second of the oracle forward on one row per host
    thread (the oracle runs one thread per row, so fewer rows than threads
    would time only part of the cores)."""
    import oracle
    n = min(oracle.default_threads(), h.shape[0])
    t0 = time.perf_counter()
    oracle.forward(h[:n], W, y[:n])
    dt = time.perf_counter() - t0
    return n * W.shape[0] * W.shape[1] / max(dt, 1e-6)


def time_oracle_sample(h, W, y, rows: int):
    """Float64 forward + backward (lse, loss, dH, full dW) on the first
    `rows` rows; returns seconds."""
    import oracle
    t0 = time.perf_counter()
    oracle.forward(h[:rows], W, y[:rows])
    oracle.backward(h[:rows], W, y[:rows], dloss=1.0)
    return time.perf_counter() - t0


def sample_rows_for(seconds: float, rate: float, wl) -> int:
    per_row = 4.0 * wl.H * wl.V  # fwd + recompute + dH + dW multiply-adds
    return int(max(1, min(wl.L, round(seconds * rate / per_row))))


def cpu_inputs(wl, rows: int):
    """The workload's distributions on the CPU: W whole, h/labels `rows`."""
    from chunked_lm_head_gemm_gb300.inputs import (make_hidden, make_labels,
                                                   make_weight)
    sub = wl.with_rows(rows)
    return make_hidden(sub, 0, "cpu"), make_weight(wl, 0, "cpu"), \
        make_labels(sub, 0)


def cpu_baseline(wl, h_cpu, W_cpu, y_cpu, target_s: float = 20.0) -> dict:
    import oracle
    oracle.build()
    rate = _oracle_rate_macs(h_cpu, W_cpu, y_cpu)
    rows = min(h_cpu.shape[0], sample_rows_for(target_s, rate, wl))
    t = time_oracle_sample(h_cpu, W_cpu, y_cpu, rows)
    return {"value": rows / t, "unit": "tokens/s",
            "cores": oracle.default_threads(), "kind": "oracle",
            "sample": (f"first {rows} of {wl.L} rows of {wl.name} (full "
                       f"H={wl.H}, V={wl.V}); float64 forward + backward "
                       f"(lse, loss, dH, full dW) in {t:.1f} s; tokens/s = "
                       f"sample rows / time"),
            "extrapolated_full_step_s": wl.L * t / rows,
            "extrapolated_note": ("not measured: the sample's time scaled to "
                                  "all rows (the float64 dW pass grows with "
                                  "the rows like the rest)")}


def run_reference(args, wl) -> dict:
    import oracle
    oracle.build()
    probe_rows = min(wl.L, oracle.default_threads())
    h, W, y = cpu_inputs(wl, probe_rows)
    rate = _oracle_rate_macs(h, W, y)
    # bounded sample per step: the whole --warmup + --steps run ~2 minutes
    per_step_s = min(10.0, 120.0 / max(1, args.steps + args.warmup))
    rows = sample_rows_for(per_step_s, rate, wl)
    h, W, y = cpu_inputs(wl, rows)
    for _ in range(args.warmup):
        time_oracle_sample(h, W, y, rows)
    times = [time_oracle_sample(h, W, y, rows) for _ in range(args.steps)]
    t = statistics.median(times)
    value = rows / t
    cores = oracle.default_threads()
    sample = (f"first {rows} of {wl.L} rows of {wl.name} (full H={wl.H}, "
              f"V={wl.V}) per step; float64 forward + backward (lse, loss, "
              f"dH, full dW); tokens/s = rows / median step time")
    return {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "L": wl.L, "H": wl.H, "V": wl.V,
                   "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------

def time_vocab_slice(lce, B, h, W, y, P: int, chunk: int, steps: int,
                     warmup: int) -> dict:
    """One process's share of a P-way vocabulary-parallel step: the forward
    statistics of its V/P slice of the head, the merge of P slices'
    statistics (this slice's, repeated: the merge reads P of them either
    way), and the slice's backward. The all-gather and all-reduce between
    processes are not part of it (one GPU)."""
    import torch
    L, H = h.shape
    V = W.shape[0]
    Vs = (V + P - 1) // P
    Ws = W[:Vs]
    ws = lce.alloc_workspace(L, H, Vs, h.dtype, chunk, h.device)
    d = torch.ones(1, dtype=torch.float32, device=h.device)

    def step():
        m, s, zy = B.forward_slice(h, Ws, y, 0, V, workspace=ws)
        st = torch.stack([m, s, zy]).unsqueeze(0).expand(P, 3, L)
        loss, lse = B.combine_slices(st[:, 0].contiguous(),
                                     st[:, 1].contiguous(),
                                     st[:, 2].contiguous(), y, V)
        B.backward_slice(h, Ws, y, lse, d, 0, V, chunk_rows=chunk,
                         workspace=ws)

    wsx = B.slice_exp_workspace(L, H, Vs, h.dtype, h.device)

    def step_exp():
        m, s, zy = B.forward_slice_exp(h, Ws, y, 0, V, wsx)
        st = torch.stack([m, s, zy]).unsqueeze(0).expand(P, 3, L)
        loss, lse = B.combine_slices(st[:, 0].contiguous(),
                                     st[:, 1].contiguous(),
                                     st[:, 2].contiguous(), y, V)
        B.backward_slice_exp(h, Ws, y, lse, d, 0, V, wsx)

    def timed_ms(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        if lce.get_error() != 0:
            raise RuntimeError("device error in the vocabulary-slice step")
        return e0.elapsed_time(e1) / steps

    ms = timed_ms(step)
    ms_exp = timed_ms(step_exp)
    del wsx
    return {"shards": P, "slice_rows": Vs, "ms_per_step_per_process": ms,
            "tokens_per_s": L / (ms / 1e3),
            "tflops_per_process_executed": 8.0 * L * H * Vs / (ms / 1e3)
            / 1e12,
            "keep_exp": {"ms_per_step_per_process": ms_exp,
                         "tokens_per_s": L / (ms_exp / 1e3),
                         "tflops_per_process_executed":
                             6.0 * L * H * Vs / (ms_exp / 1e3) / 1e12},
            "note": "forward slice + merge + recomputing backward slice "
                    "(keep_exp: the slice's exponentials kept between the "
                    "two, no recompute); collectives not timed"}


def time_torch_chunked(h, W, y, chunk_rows: int, steps: int,
                       warmup: int) -> dict:
    """Context only, never part of the library: the pages' own chunked
    scheme ("Training Beyond 1M Tokens", section "The massive logits matrix:
    chunk it") in eager PyTorch on the same GPU -- per chunk of rows, cuBLAS
    bf16 logits, fp32 cross-entropy, autograd backward at once (no
    recompute), dW accumulated in W's dtype by autograd."""
    import torch
    import torch.nn.functional as F
    L = h.shape[0]
    n = (y != -100).sum().clamp(min=1).to(torch.float32)
    Wl = W.detach().requires_grad_(True)
    dH = torch.empty_like(h)

    def step():
        Wl.grad = None
        total = torch.zeros((), dtype=torch.float32, device=h.device)
        for c0 in range(0, L, chunk_rows):
            c1 = min(L, c0 + chunk_rows)
            hc = h[c0:c1].detach().requires_grad_(True)
            z = F.linear(hc, Wl).float()
            lc = F.cross_entropy(z, y[c0:c1], ignore_index=-100,
                                 reduction="sum") / n
            lc.backward()
            dH[c0:c1] = hc.grad
            total += lc.detach()
        return total

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    H, V = h.shape[1], W.shape[0]
    return {"impl": "eager PyTorch, autograd per chunk (context only)",
            "chunk_rows": chunk_rows, "ms_per_step": ms,
            "tokens_per_s": L / (ms / 1e3),
            "tflops_model": 6.0 * L * H * V / (ms / 1e3) / 1e12,
            "steps": steps, "warmup": warmup}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="lce", choices=["lce", "reference"])
    ap.add_argument("--config", default="qwen3-8b")
    ap.add_argument("--rows", type=int, default=0,
                    help="override L (a row slice of the workload)")
    ap.add_argument("--vocab", type=int, default=0,
                    help="override V (a reduced vocabulary, for profiling "
                         "one contraction on a small device footprint)")
    ap.add_argument("--chunk-rows", type=int, default=0)
    ap.add_argument("--label-smoothing", type=float, default=0.0,
                    help="time the loss variant with this label smoothing "
                         "(lce_*_ex calls; 0 = the plain loss)")
    ap.add_argument("--z-loss", type=float, default=0.0,
                    help="time the loss variant with this z-loss "
                         "coefficient (0 = none)")
    ap.add_argument("--mode", default="fused", choices=["separate", "fused"])
    ap.add_argument("--only-mode", action="store_true",
                    help="time only --mode (profiling runs)")
    ap.add_argument("--workload", default="lce", choices=["lce", "mlp"])
    ap.add_argument("--cta-pair", type=int, default=-1, choices=[-1, 0, 1],
                    help="contractions on CTA pairs (1) or single CTAs (0); "
                         "-1 keeps the library default")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--vocab-shards", type=int, default=0, metavar="P",
                    help="also time one process's share of a P-way "
                         "vocabulary-parallel step (its V/P slice; the "
                         "collectives are not timed)")
    ap.add_argument("--layout-sweep", default="", metavar="M,N,K",
                    help="time the library's contraction D = A B on M,N,K in "
                         "its four operand layouts (A, B K-major or "
                         "MN-major) and print one JSON line instead of the "
                         "benchmark")
    ap.add_argument("--forward-static", action="store_true",
                    help="time lce_forward_static against lce_forward on "
                         "the workload (forward only) and print one JSON "
                         "line instead of the benchmark")
    ap.add_argument("--comparator", type=int, default=0, metavar="ROWS",
                    help="also time the pages' chunked scheme in eager "
                         "PyTorch with ROWS-row chunks (context only)")
    args = ap.parse_args()

    if args.layout_sweep:
        return layout_sweep(args)
    if args.forward_static:
        return forward_static(args)
    if args.workload == "mlp":
        return bench_mlp(args)
    from chunked_lm_head_gemm_gb300.inputs import WORKLOADS
    wl = WORKLOADS[args.config]
    if args.rows:
        wl = wl.with_rows(args.rows)
    if args.vocab:
        import dataclasses
        wl = dataclasses.replace(wl, V=args.vocab,
                                 name=f"{wl.name}[V={args.vocab}]")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, wl)), flush=True)
        return

    import torch
    import chunked_lm_head_gemm_gb300 as lce
    from chunked_lm_head_gemm_gb300 import _binding as B
    from chunked_lm_head_gemm_gb300.inputs import make_inputs

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    lce.load()
    if args.cta_pair >= 0:
        B.set_cta_pair(bool(args.cta_pair))

    def barrier():
        if dist is not None:
            dist.barrier()

    h, W, y = make_inputs(wl, seed=0, device=dev)
    L, H, V = wl.L, wl.H, wl.V
    chunk = args.chunk_rows or lce.default_chunk_rows(L, H, V)
    ws = lce.alloc_workspace(L, H, V, h.dtype, chunk, dev)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    lse = torch.empty(L, dtype=torch.float32, device=dev)
    dH = torch.empty_like(h)
    dW = torch.empty(V, H, dtype=torch.float32, device=dev)
    dloss = torch.ones(1, dtype=torch.float32, device=dev)

    variant = dict(label_smoothing=args.label_smoothing, z_loss=args.z_loss)

    def step_separate():
        lce.forward(h, W, y, workspace=ws, loss_out=loss, lse_out=lse,
                    **variant)
        lce.backward(h, W, y, lse, dloss, chunk_rows=chunk, workspace=ws,
                     dH_out=dH, dW_out=dW, **variant)

    def step_fused():
        lce.forward_backward(h, W, y, chunk_rows=chunk, workspace=ws,
                             loss_out=loss, lse_out=lse, dH_out=dH,
                             dW_out=dW, **variant)
        lce.scale_gradients(dH, dW, dloss)

    steps = {"separate": step_separate, "fused": step_fused}
    step = steps[args.mode]

    in_bytes = h.numel() * h.element_size() + W.numel() * W.element_size()
    flush = None
    if in_bytes < 4 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def timed(step_fn, with_clocks):
        """W warm-up steps, then exactly K steps between CUDA events, the
        library's per-kernel events on; returns (max-over-ranks ms, kernel
        stats, clocks)."""
        for _ in range(args.warmup):
            step_fn()
        torch.cuda.synchronize()
        st = lce.get_error()
        if st != 0:
            raise RuntimeError(f"device error status {st} during warm-up")
        clocks = ClockSampler(local) if with_clocks else None
        if clocks:
            clocks.start()
        barrier()
        torch.cuda.synchronize()
        B.profile_start()
        if flush is None:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.steps):
                step_fn()
            e1.record()
            torch.cuda.synchronize()
            elapsed_ms = e0.elapsed_time(e1)
        else:
            elapsed_ms = 0.0
            for _ in range(args.steps):
                flush.fill_(1.0)  # evict h and W from L2 between steps
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                step_fn()
                e1.record()
                torch.cuda.synchronize()
                elapsed_ms += e0.elapsed_time(e1)
        stats = B.profile_stop()
        barrier()
        clk = clocks.stop() if clocks else None
        st = lce.get_error()
        if st != 0:
            raise RuntimeError(f"device error status {st} in the timed region")
        tt = torch.tensor([elapsed_ms], dtype=torch.float64, device=dev)
        if dist is not None:
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        return tt.item(), stats, clk

    modes = {}
    phases = {}
    if not args.only_mode:
        for m in steps:
            if m != args.mode:
                ms, _, _ = timed(steps[m], False)
                modes[m] = ms
        # the separate path's two calls on their own: forward (logits pass,
        # loss) and backward (recompute, dH, dW) from the forward's lse
        def step_fwd():
            lce.forward(h, W, y, workspace=ws, loss_out=loss, lse_out=lse,
                        **variant)

        def step_bwd():
            lce.backward(h, W, y, lse, dloss, chunk_rows=chunk, workspace=ws,
                         dH_out=dH, dW_out=dW, **variant)
        for name, fn in (("forward", step_fwd), ("backward", step_bwd)):
            ms, _, _ = timed(fn, False)
            phases[name] = {"ms": ms / args.steps,
                            "tflops": 2.0 * (1 if name == "forward" else 3)
                            * L * H * V / (ms / args.steps / 1e3) / 1e12}
    elapsed_ms, stats, clk = timed(step, True)
    modes[args.mode] = elapsed_ms
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=dev)
    t_max_s = t.item() / 1e3
    tokens = float(L) * args.steps * world
    value = tokens / t_max_s
    ms_per_step = t.item() / args.steps
    peaks, peak_src = load_peaks()
    per_gpu_s = t_max_s / args.steps
    tf_model = 6.0 * L * H * V / per_gpu_s / 1e12
    exec_flops = (8.0 if args.mode == "separate" else 6.0) * L * H * V
    tf_exec = exec_flops / per_gpu_s / 1e12
    modes_out = {m: {"ms_per_step": ms / args.steps,
                     "tokens_per_s": float(L) * world * args.steps / (ms / 1e3),
                     "tflops_model": 6.0 * L * H * V / (ms / args.steps / 1e3)
                     / 1e12}
                 for m, ms in modes.items()}
    if phases and "separate" in modes_out:
        modes_out["separate"]["phases"] = phases

    # dominant kernel: largest total event time in the timed region
    kernels = {}
    total_k_ms = sum(v[1] for v in stats.values()) or 1.0
    for name, (n, ms, fl) in stats.items():
        kernels[name] = {"launches": n, "ms_per_launch": ms / n,
                         "share": ms / total_k_ms,
                         "tflops": (fl / (ms / 1e3) / 1e12) if fl else None}
    dom = max(stats.items(), key=lambda kv: kv[1][1])
    dname, (dn, dms, dfl) = dom
    peak_t = peaks["bf16_tflops_sustained"]
    achieved = dfl / (dms / 1e3) / 1e12
    traffic = load_traffic(dname, wl.name)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak_t,
                "unit": "TFLOP/s", "frac": achieved / peak_t,
                "traffic": traffic, "kernel": dname,
                "flops_per_launch": dfl / dn,
                "peak_source": f"bf16 sustained, {peak_src}"}
    gpu_launches = int(sum(v[0] for v in stats.values()))

    # ---- end to end: pinned host in, results out, inside the timed region --
    # Every step copies its inputs (h, W, labels) from pinned host memory and
    # reads its results (loss, dH, dW) back into pinned host memory. Two
    # device buffer sets and two copy streams let step i+1's inputs arrive
    # and step i-1's results leave while step i computes ("pipelined");
    # "sequential_value" is the same loop with every copy on the compute
    # stream.
    e2e = None
    if not args.no_e2e:
        pin = dict(pin_memory=True)
        h_host = torch.empty(h.shape, dtype=h.dtype, **pin)
        W_host = torch.empty(W.shape, dtype=W.dtype, **pin)
        y_host = torch.empty(y.shape, dtype=y.dtype, **pin)
        h_host.copy_(h)
        W_host.copy_(W)
        y_host.copy_(y)
        loss_host = torch.empty((), dtype=torch.float32, **pin)
        dH_host = torch.empty(dH.shape, dtype=dH.dtype, **pin)
        dW_host = torch.empty(dW.shape, dtype=dW.dtype, **pin)
        bufs = [dict(h=h, W=W, y=y, loss=loss, lse=lse, dH=dH, dW=dW),
                dict(h=torch.empty_like(h), W=torch.empty_like(W),
                     y=torch.empty_like(y), loss=torch.empty_like(loss),
                     lse=torch.empty_like(lse), dH=torch.empty_like(dH),
                     dW=torch.empty_like(dW))]

        def compute(b):
            if args.mode == "fused":
                lce.forward_backward(b["h"], b["W"], b["y"], chunk_rows=chunk,
                                     workspace=ws, loss_out=b["loss"],
                                     lse_out=b["lse"], dH_out=b["dH"],
                                     dW_out=b["dW"])
                lce.scale_gradients(b["dH"], b["dW"], dloss)
            else:
                lce.forward(b["h"], b["W"], b["y"], workspace=ws,
                            loss_out=b["loss"], lse_out=b["lse"])
                lce.backward(b["h"], b["W"], b["y"], b["lse"], dloss,
                             chunk_rows=chunk, workspace=ws, dH_out=b["dH"],
                             dW_out=b["dW"])

        def copy_in(b):
            b["h"].copy_(h_host, non_blocking=True)
            b["W"].copy_(W_host, non_blocking=True)
            b["y"].copy_(y_host, non_blocking=True)

        def copy_out(b):
            loss_host.copy_(b["loss"], non_blocking=True)
            dH_host.copy_(b["dH"], non_blocking=True)
            dW_host.copy_(b["dW"], non_blocking=True)

        def run_sequential(nsteps):
            for _ in range(nsteps):
                copy_in(bufs[0])
                compute(bufs[0])
                copy_out(bufs[0])

        s_in = torch.cuda.Stream(device=dev)
        s_out = torch.cuda.Stream(device=dev)
        comp = torch.cuda.current_stream(dev)

        def run_pipelined(nsteps):
            ev_in = [torch.cuda.Event() for _ in range(nsteps)]
            ev_done = [torch.cuda.Event() for _ in range(nsteps)]
            ev_out = [torch.cuda.Event() for _ in range(nsteps)]
            start = torch.cuda.Event()
            start.record(comp)
            s_in.wait_event(start)
            s_out.wait_event(start)
            for i in range(nsteps):
                b = bufs[i % 2]
                with torch.cuda.stream(s_in):
                    if i >= 2:  # step i-2 has finished reading this set
                        s_in.wait_event(ev_done[i - 2])
                    copy_in(b)
                    ev_in[i].record(s_in)
                comp.wait_event(ev_in[i])
                if i >= 2:  # step i-2's results have left this set
                    comp.wait_event(ev_out[i - 2])
                compute(b)
                ev_done[i].record(comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_done[i])
                    copy_out(b)
                    ev_out[i].record(s_out)
            comp.wait_event(ev_out[nsteps - 1])

        def time_e2e(fn):
            fn(1)
            torch.cuda.synchronize()
            barrier()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            wall0 = time.perf_counter()
            e0.record()
            fn(args.steps)
            e1.record()
            torch.cuda.synchronize()
            wall = time.perf_counter() - wall0
            te = torch.tensor([e0.elapsed_time(e1)], dtype=torch.float64,
                              device=dev)
            if dist is not None:
                dist.all_reduce(te, op=dist.ReduceOp.MAX)
            assert torch.isfinite(loss_host).item()
            return tokens / (te.item() / 1e3), wall

        seq_value, seq_wall = time_e2e(run_sequential)
        pipe_value, pipe_wall = time_e2e(run_pipelined)
        st = lce.get_error()
        if st != 0:
            raise RuntimeError(f"device error status {st} in the e2e loop")
        e2e = {"value": pipe_value, "unit": "tokens/s",
               "h2d_bytes_per_step": int(h_host.nbytes + W_host.nbytes +
                                         y_host.nbytes),
               "d2h_bytes_per_step": int(loss_host.nbytes + dH_host.nbytes +
                                         dW_host.nbytes),
               "pipelined": True, "wall_s": pipe_wall,
               "sequential_value": seq_value, "sequential_wall_s": seq_wall}
        del h_host, W_host, dH_host, dW_host, bufs

    vocab_par = None
    if args.vocab_shards >= 1:
        vocab_par = time_vocab_slice(lce, B, h, W, y, args.vocab_shards,
                                     chunk, args.steps, args.warmup)

    comparator = None
    if args.comparator:
        comparator = time_torch_chunked(h, W, y, args.comparator, 2, 1)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows = min(L, 512)
        hc = h[:rows].cpu()
        yc = y[:rows].cpu()
        Wc = W.cpu()
        cpu = cpu_baseline(wl, hc, Wc, yc)

    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": wl.name, "L": L, "H": H, "V": V,
                       "inputs": wl.dtype, "chunk_rows": chunk,
                       "mode": args.mode,
                       **({"label_smoothing": args.label_smoothing,
                           "z_loss": args.z_loss}
                          if args.label_smoothing or args.z_loss else {}),
                       "cta_pair": B.get_cta_pair(),
                       "parallelism": "replicas" if world > 1 else "single",
                       "l2": ("inputs larger than L2, no flush" if flush is None
                              else "L2 flushed between steps (not timed)")},
            "tflops_model": tf_model, "tflops_executed": tf_exec,
            "frac_of_bf16_peak": tf_model / peak_t,
            "peak_note": (f"6LHV model flops per GPU vs {peak_t} TFLOP/s bf16 "
                          f"sustained ({peak_src}); the executed basis is "
                          "8LHV for the separate path (the backward "
                          "recomputes the logits), 6LHV for the fused path"),
            "modes": modes_out,
            "roofline": roofline, "kernels": kernels,
            "gpu_launches": gpu_launches, "clocks": clk, "e2e": e2e,
            "cpu_baseline": cpu,
            "peak_extra_bytes": int(ws.numel()),
        }
        ctx = PAGES_STEP.get(wl.name.split("[")[0])
        if ctx and not args.rows:
            out["pages_context"] = dict(
                ctx, loss_share_of_step=(ms_per_step / 1e3) / ctx["s_per_step"],
                note=("the pages' whole training step, of which this "
                      "workload is one GPU's shard of the loss; context "
                      "only; loss_share_of_step = this fwd+bwd time on one "
                      "GB300 over that step time"))
        if comparator:
            out["comparator"] = comparator
        if vocab_par:
            out["vocab_parallel"] = vocab_par
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def forward_static(args):
    """lce_forward_static (fixed scratch inside the library, single-CTA
    contraction, no wave pacing) against lce_forward (caller workspace,
    the default contraction variant, paced) on the same inputs, interleaved:
    median ms per call from CUDA events; one JSON line."""
    import ctypes
    import torch
    import chunked_lm_head_gemm_gb300 as lce
    from chunked_lm_head_gemm_gb300.inputs import WORKLOADS, make_inputs
    wl = WORKLOADS[args.config]
    if args.rows:
        wl = wl.with_rows(args.rows)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lib = lce.load()
    h, W, y = make_inputs(wl, seed=0, device=dev)
    L, H, V = wl.L, wl.H, wl.V
    ws = lce.alloc_workspace(L, H, V, h.dtype, 0, dev)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    lse = torch.empty(L, dtype=torch.float32, device=dev)

    def static():
        st = lib.lce_forward_static(
            ctypes.c_void_p(h.data_ptr()), ctypes.c_void_p(W.data_ptr()),
            ctypes.c_void_p(y.data_ptr()), L, H, V, -100,
            ctypes.c_void_p(loss.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        if st != 0:
            raise RuntimeError(lib.lce_last_cuda_error().decode())

    def workspace():
        lce.forward(h, W, y, workspace=ws, loss_out=loss, lse_out=lse)

    calls = {"lce_forward_static": static, "lce_forward": workspace}
    for _ in range(args.warmup):
        for f in calls.values():
            f()
    torch.cuda.synchronize()
    ms = {k: [] for k in calls}
    for _ in range(args.steps):
        for k, f in calls.items():
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            f()
            e1.record()
            torch.cuda.synchronize()
            ms[k].append(e0.elapsed_time(e1))
    if lce.get_error() != 0:
        raise RuntimeError("device error status in the static-forward timing")
    flops = 2.0 * L * H * V
    out = {k: {"ms_median": statistics.median(v),
               "tflops": flops / statistics.median(v) / 1e9}
           for k, v in ms.items()}
    print(json.dumps({"forward_static": out, "workload": wl.name,
                      "steps": args.steps}), flush=True)


def layout_sweep(args):
    """The contraction D[M,N] = A[M,K] B[K,N] (bf16, fp32 out) through the
    library's test hook in its four operand layouts, interleaved, on the
    contraction variant in use: TFLOP/s per layout from CUDA events over
    --steps launches each, after --warmup; one JSON line."""
    import torch
    import chunked_lm_head_gemm_gb300 as lce
    from chunked_lm_head_gemm_gb300 import _binding as B
    M, N, K = (int(x) for x in args.layout_sweep.split(","))
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lce.load()
    if args.cta_pair >= 0:
        B.set_cta_pair(bool(args.cta_pair))
    g = torch.Generator(device=dev).manual_seed(0)
    ops = {}
    for a_mn in (False, True):
        for b_mn in (False, True):
            A = torch.randn(*((K, M) if a_mn else (M, K)), generator=g,
                            device=dev).to(torch.bfloat16)
            Bm = torch.randn(*((K, N) if b_mn else (N, K)), generator=g,
                             device=dev).to(torch.bfloat16)
            ops[(a_mn, b_mn)] = (A, Bm)
    ms = {k: [] for k in ops}
    for _ in range(args.warmup):
        for (a_mn, b_mn), (A, Bm) in ops.items():
            B.tc_gemm(A, Bm, M, N, K, a_mn, b_mn)
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    for _ in range(args.steps):
        for (a_mn, b_mn), (A, Bm) in ops.items():
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            B.tc_gemm(A, Bm, M, N, K, a_mn, b_mn)
            e1.record()
            torch.cuda.synchronize()
            ms[(a_mn, b_mn)].append(e0.elapsed_time(e1))
    clk = clocks.stop()
    if lce.get_error() != 0:
        raise RuntimeError("device error status in the layout sweep")
    flops = 2.0 * M * N * K
    name = {(False, False): "A K-major, B K-major",
            (False, True): "A K-major, B MN-major",
            (True, False): "A MN-major, B K-major",
            (True, True): "A MN-major, B MN-major"}
    out = {}
    for k, v in ms.items():
        med = statistics.median(v)
        out[name[k]] = {"ms_median": med, "tflops": flops / med / 1e9}
    print(json.dumps({"layout_sweep": out, "M": M, "N": N, "K": K,
                      "steps": args.steps, "cta_pair": B.get_cta_pair(),
                      "clocks": clk}), flush=True)


def bench_mlp(args):
    """The sequence-tiled gated MLP: y = (silu(x Wg^T) * (x Wu^T)) Wd^T,
    forward + backward per step on one GPU (replicas under torchrun)."""
    import torch
    import chunked_lm_head_gemm_gb300 as lce
    from chunked_lm_head_gemm_gb300 import _binding as B
    from chunked_lm_head_gemm_gb300.inputs import MLP_WORKLOADS, make_mlp_inputs
    name = args.config if args.config.endswith("-mlp") else "qwen3-8b-mlp"
    wl = MLP_WORKLOADS[name]
    if args.rows:
        wl = wl.with_rows(args.rows)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    metric = "sequence-tiled gated MLP fwd+bwd tokens/s"
    if args.impl == "reference":
        if rank == 0:
            import oracle
            from chunked_lm_head_gemm_gb300.inputs import make_mlp_inputs as mk
            oracle.build()
            rows = 8
            x, Wg, Wu, Wd, dy = mk(wl.with_rows(rows), 0, "cpu")
            for _ in range(args.warmup):
                oracle.mlp(x, Wg, Wu, Wd, dy)
            times = []
            for _ in range(args.steps):
                t0 = time.perf_counter()
                oracle.mlp(x, Wg, Wu, Wd, dy)
                times.append(time.perf_counter() - t0)
            t = statistics.median(times)
            v = rows / t
            print(json.dumps({
                "impl": "reference", "metric": metric, "value": v,
                "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": t * 1e3,
                "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": wl.name, "L": wl.L, "H": wl.H,
                           "I": wl.I, "sample_rows": rows},
                "cpu_baseline": {"value": v, "unit": "tokens/s",
                                 "cores": oracle.default_threads(),
                                 "kind": "oracle",
                                 "sample": f"{rows} rows per step"},
                "e2e": {"value": v, "unit": "tokens/s",
                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
                flush=True)
        return
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    lce.load()
    if args.cta_pair >= 0:
        B.set_cta_pair(bool(args.cta_pair))
    x, Wg, Wu, Wd, dy = make_mlp_inputs(wl, seed=0, device=dev)
    L, H, I = wl.L, wl.H, wl.I
    chunk = args.chunk_rows
    ws = torch.empty(lce.mlp_workspace_size(L, H, I, chunk),
                     dtype=torch.uint8, device=dev)
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    dWg = torch.empty(I, H, dtype=torch.float32, device=dev)
    dWu = torch.empty(I, H, dtype=torch.float32, device=dev)
    dWd = torch.empty(H, I, dtype=torch.float32, device=dev)

    def step():
        lce.mlp_forward(x, Wg, Wu, Wd, chunk, ws, y)
        lce.mlp_backward(x, Wg, Wu, Wd, dy, chunk, ws, dx, dWg, dWu, dWd)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if lce.get_error() != 0:
        raise RuntimeError("device error during warm-up")
    clocks = ClockSampler(local)
    clocks.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    B.profile_start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    stats = B.profile_stop()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    if lce.get_error() != 0:
        raise RuntimeError("device error in the timed region")
    t = torch.tensor([e0.elapsed_time(e1)], dtype=torch.float64, device=dev)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    per_step = t.item() / 1e3 / args.steps
    peaks, peak_src = load_peaks()
    peak_t = peaks["bf16_tflops_sustained"]
    kernels = {}
    total_k_ms = sum(v[1] for v in stats.values()) or 1.0
    for kname, (n, ms, fl) in stats.items():
        kernels[kname] = {"launches": n, "ms_per_launch": ms / n,
                          "share": ms / total_k_ms,
                          "tflops": (fl / (ms / 1e3) / 1e12) if fl else None}
    dname, (dn, dms, dfl) = max(stats.items(), key=lambda kv: kv[1][1])
    achieved = dfl / (dms / 1e3) / 1e12
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        rows = 16
        t0 = time.perf_counter()
        oracle.mlp(x[:rows].cpu(), Wg.cpu(), Wu.cpu(), Wd.cpu(),
                   dy[:rows].cpu())
        tc = time.perf_counter() - t0
        cpu = {"value": rows / tc, "unit": "tokens/s",
               "cores": oracle.default_threads(), "kind": "oracle",
               "sample": f"first {rows} rows, float64 forward + backward "
                         f"(y, dx, dWg, dWu, dWd) in {tc:.1f} s"}
    if rank == 0:
        print(json.dumps({
            "metric": metric, "value": L * world / per_step,
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": per_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "L": L, "H": H, "I": I,
                       "chunk_rows": chunk or "default",
                       "cta_pair": B.get_cta_pair(),
                       "l2": "inputs larger than L2, no flush"},
            "tflops_model": 18.0 * L * H * I / per_step / 1e12,
            "tflops_executed": 22.0 * L * H * I / per_step / 1e12,
            "peak_note": (f"18LHI model flops (22LHI executed: the backward "
                          f"recomputes gate/up) vs {peak_t} TFLOP/s bf16 "
                          f"sustained ({peak_src})"),
            "roofline": {"bound": "tensor", "achieved": achieved,
                         "peak": peak_t, "unit": "TFLOP/s",
                         "frac": achieved / peak_t, "traffic": None,
                         "kernel": dname, "flops_per_launch": dfl / dn},
            "kernels": kernels,
            "gpu_launches": int(sum(v[0] for v in stats.values())),
            "clocks": clk, "cpu_baseline": cpu}), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
