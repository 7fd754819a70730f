"""Wave pacing of the contractions is only a hint about timing: with it on
or off, every path gives bit-identical loss, lse and gradients (fixed
reduction orders), on both contraction variants, on a case with many waves
of tiles per launch and several row chunks."""
import pytest
import torch

import chunked_lm_head_gemm_gb300 as lce
from chunked_lm_head_gemm_gb300 import _binding as B
from chunked_lm_head_gemm_gb300.inputs import WORKLOADS, make_inputs
from tests.gpu_util import MODES, PAIRS, cta_pair, require_gpu

pytestmark = pytest.mark.gpu


def _run(h, W, y, mode):
    if mode == "fused":
        return lce.forward_backward(h, W, y, chunk_rows=1024)
    loss, lse = lce.forward(h, W, y)
    dH, dW = lce.backward(h, W, y, lse, torch.ones(1, device=h.device),
                          chunk_rows=1024)
    return loss, lse, dH, dW


@pytest.mark.parametrize("pair", PAIRS, ids=lambda v: "pair" if v else "cta")
@pytest.mark.parametrize("mode", MODES)
def test_pacing_does_not_change_results(mode, pair):
    dev = require_gpu()
    wl = WORKLOADS["qwen3-0.6b"].with_rows(3000)
    h, W, y = make_inputs(wl, seed=4, device=dev)
    before = B.get_wave_sync()
    try:
        with cta_pair(pair):
            B.set_wave_sync(True)
            on = _run(h, W, y, mode)
            B.set_wave_sync(False)
            off = _run(h, W, y, mode)
    finally:
        B.set_wave_sync(before)
    assert lce.get_error() == 0
    for a, b in zip(on, off):
        assert torch.equal(a, b)


@pytest.mark.parametrize("pair", PAIRS, ids=lambda v: "pair" if v else "cta")
def test_pacing_does_not_change_mlp_results(pair):
    """The gated MLP's contractions are paced too (with every other
    contraction, their tiles grouped by 8 columns): on and off give the same
    bits, on a case with several row chunks and many tiles per launch."""
    dev = require_gpu()
    from chunked_lm_head_gemm_gb300.inputs import MLP_WORKLOADS, make_mlp_inputs
    wl = MLP_WORKLOADS["qwen3-0.6b-mlp"].with_rows(2560)
    x, Wg, Wu, Wd, dy = make_mlp_inputs(wl, seed=6, device=dev)
    before = B.get_wave_sync()
    out = {}
    try:
        with cta_pair(pair):
            for on in (True, False):
                B.set_wave_sync(on)
                y = lce.mlp_forward(x, Wg, Wu, Wd, chunk_rows=1024)
                out[on] = (y,) + lce.mlp_backward(x, Wg, Wu, Wd, dy,
                                                  chunk_rows=1024)
    finally:
        B.set_wave_sync(before)
    assert lce.get_error() == 0
    for a, b in zip(out[True], out[False]):
        assert torch.equal(a, b)
