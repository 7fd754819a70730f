"""The tensor-core building block (tcgen05 + TMA, every operand layout, on
single CTAs and on CTA pairs) against a plain fp32 matmul of the same bf16
values."""
import pytest
import torch

from tests.gpu_util import PAIRS, rel_fro, require_gpu, to64

pytestmark = pytest.mark.gpu

SHAPES = [(128, 256, 64), (200, 264, 136), (384, 512, 1024), (64, 8, 8),
          (1000, 776, 520)]


@pytest.mark.parametrize("pair", PAIRS, ids=lambda v: "pair" if v else "cta")
@pytest.mark.parametrize("a_mn", [False, True])
@pytest.mark.parametrize("b_mn", [False, True])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_layouts(a_mn, b_mn, M, N, K, pair):
    dev = require_gpu()
    from chunked_lm_head_gemm_gb300 import _binding as B
    g = torch.Generator(device=dev)
    g.manual_seed(M * 7 + N * 3 + K)
    A = torch.randn(M, K, generator=g, device=dev).to(torch.bfloat16)
    Bm = torch.randn(K, N, generator=g, device=dev).to(torch.bfloat16)
    A_in = A.t().contiguous() if a_mn else A
    B_in = Bm.contiguous() if b_mn else Bm.t().contiguous()
    before = B.get_cta_pair()
    B.set_cta_pair(pair)
    try:
        D = B.tc_gemm(A_in, B_in, M, N, K, a_mn, b_mn)
        assert B.get_error() == 0
    finally:
        B.set_cta_pair(before)
    ref = A.double() @ Bm.double()
    assert rel_fro(to64(D), to64(ref)) < 1e-5
