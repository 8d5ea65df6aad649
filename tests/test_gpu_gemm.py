"""The tensor-core GEMM engine against float64 products of the same operands.

Covers every operand precision, all four transpose combinations (K-major and
MN-major shared-memory operands), the 128- and 256-wide tile paths and a ragged
multi-tile size (B = 384: three M tiles, three 128-wide N tiles, twelve TF32
k-blocks)."""

import pytest
import torch

from tests.helpers import library, rel_fro_blocks, require_gpu, rna_tf32, split_tf32, to64

pytestmark = pytest.mark.gpu


def operands(x, prec):
    """(hi, lo, exact float64 value the tensor core multiplies)."""
    if prec == "tf32":
        h = rna_tf32(x)
        return h, None, to64(h)
    if prec == "3xtf32":
        h, l = split_tf32(x)
        return h, l, to64(x)
    dt = torch.float16 if prec == "fp16" else torch.bfloat16
    h = x.to(dt)
    return h, None, to64(h)


@pytest.mark.parametrize("prec", ["tf32", "3xtf32", "fp16", "bf16"])
@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("b", [128, 256, 384])
def test_gemm_matches_float64(prec, ta, tb, b):
    require_gpu()
    dr = library()
    n = 3
    g = torch.Generator(device="cuda")
    g.manual_seed(1000 * b + 10 * ta + tb)
    A = torch.randn((n, b, b), generator=g, device="cuda")
    B = torch.randn((n, b, b), generator=g, device="cuda")
    Ah, Al, A64 = operands(A, prec)
    Bh, Bl, B64 = operands(B, prec)
    C = dr.gemm(Ah, Bh, prec=prec, trans_a=ta, trans_b=tb, A_lo=Al, B_lo=Bl)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    opA = A64.transpose(0, 2, 1) if ta else A64
    opB = B64.transpose(0, 2, 1) if tb else B64
    ref = opA @ opB
    err = rel_fro_blocks(to64(C), ref)
    tol = 2e-5 if prec == "3xtf32" else 1e-5
    assert err.max() < tol, (prec, ta, tb, b, err)


def test_gemm_large_k_and_many_blocks():
    require_gpu()
    dr = library()
    # B = 2048 (64 k-blocks of fp16) and more tiles than SMs for a few blocks.
    for b, n in ((2048, 2), (512, 40)):
        g = torch.Generator(device="cuda")
        g.manual_seed(b + n)
        A = torch.randn((n, b, b), generator=g, device="cuda").half()
        B = torch.randn((n, b, b), generator=g, device="cuda").half()
        C = dr.gemm(A, B, prec="fp16")
        torch.cuda.synchronize()
        assert dr.device_status() == 0
        idx = [0, n // 2, n - 1]
        ref = to64(A[idx]) @ to64(B[idx])
        assert rel_fro_blocks(to64(C[idx]), ref).max() < 1e-5
