"""bench.py's reference arm on CPU: one JSON line with the contract's keys
(the float64 oracle timed on host cores on a bounded row sample), printed
by rank 0 only."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None, *args):
    env = dict(os.environ)
    env.update(extra_env or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", *args],
                       capture_output=True, text=True, env=env, cwd=ROOT,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout


def test_reference_arm_json_line(oracle_mod):
    out = _run(None, "--config", "tiny", "--steps", "2", "--warmup", "1")
    lines = [l for l in out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup",
              "ms_per_step", "higher_is_better", "scaling", "vs_baseline",
              "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny"
    assert 1 <= d["config"]["sample_rows"] <= 512
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_silent_on_other_ranks():
    out = _run({"RANK": "1", "WORLD_SIZE": "2"}, "--config", "tiny",
               "--steps", "1", "--warmup", "0", "--gpus", "2")
    assert out.strip() == ""


def test_traffic_lookup_follows_the_kernel_source(tmp_path, monkeypatch):
    """The roofline's DRAM traffic is reported only for the kernel source
    the committed capture was taken on (else null)."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    prof = tmp_path / "profiles"
    prof.mkdir()
    h = bench.source_hash()
    (prof / "traffic.json").write_text(json.dumps({
        "gemm_dW": {"qwen3-8b": {"dram_bytes_per_launch": 123.0,
                                 "source_hash": h}},
        "gemm_dH": {"qwen3-8b": {"dram_bytes_per_launch": 7.0,
                                 "source_hash": "0" * 16}}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda: h)
    assert bench.load_traffic("gemm_dW", "qwen3-8b") == 123.0
    assert bench.load_traffic("gemm_dH", "qwen3-8b") is None
    assert bench.load_traffic("gemm_dW", "qwen3-4b") is None


def test_oracle_sample_is_bounded():
    sys.path.insert(0, ROOT)
    import bench
    from chunked_lm_head_gemm_gb300.inputs import WORKLOADS
    wl = WORKLOADS["qwen3-8b"]
    # rows so that the float64 work takes about `seconds` at `rate`
    rows = bench.sample_rows_for(20.0, 4.0 * wl.H * wl.V * 3.0, wl)
    assert rows == 60
    assert bench.sample_rows_for(1e9, 1e12, wl) == wl.L
    assert bench.sample_rows_for(1e-9, 1.0, wl) == 1
