"""Argument errors, workspace errors and the bounded-wait failure path on
the GPU (no kernel is made to fault, trap or hang)."""
import pytest
import torch

from tests.gpu_util import require_gpu

pytestmark = pytest.mark.gpu


def _small(dev, L=64, H=32, V=300, dtype=torch.bfloat16):
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    h = torch.randn(L, H, generator=g, device=dev).to(dtype)
    W = (0.1 * torch.randn(V, H, generator=g, device=dev)).to(dtype)
    y = torch.randint(0, V, (L,), device=dev, generator=g)
    return h, W, y


def test_invalid_arguments_rejected_before_launch():
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    from chunked_lm_head_gemm_gb300 import _binding as B
    h, W, y = _small(dev, H=12)  # H not a multiple of 8
    with pytest.raises(lce.LCEError) as ei:
        lce.forward(h, W, y, workspace=torch.empty(1 << 20, dtype=torch.uint8,
                                                   device=dev))
    assert ei.value.status == B.LCE_ERR_INVALID_ARG
    h, W, y = _small(dev)
    with pytest.raises(lce.LCEError) as ei:
        lce.forward(h, W, y, workspace=torch.empty(256, dtype=torch.uint8,
                                                   device=dev))
    assert ei.value.status == B.LCE_ERR_WORKSPACE
    buf = torch.empty(64 * 32 + 1, dtype=torch.bfloat16, device=dev)
    hm = buf[1:].view(64, 32)  # 2-byte offset: not 16-byte aligned
    hm.copy_(h)
    with pytest.raises(lce.LCEError) as ei:
        lce.forward(hm, W, y)
    assert ei.value.status == B.LCE_ERR_INVALID_ARG
    assert lce.get_error() == 0


def test_bounded_wait_expires_and_context_survives():
    dev = require_gpu()
    import chunked_lm_head_gemm_gb300 as lce
    from chunked_lm_head_gemm_gb300 import _binding as B
    assert lce.get_error() == 0
    B.wait_timeout_probe(20_000_000)  # 20 ms on a barrier nothing signals
    assert lce.get_error() == B.LCE_ERR_TIMEOUT
    assert lce.get_error() == 0
    h, W, y = _small(dev)
    loss, lse = lce.forward(h, W, y)
    assert torch.isfinite(loss).item()
    assert lce.get_error() == 0
