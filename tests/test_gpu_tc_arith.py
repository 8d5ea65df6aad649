"""The library's TF32 / 3xTF32 GEMM against the tensor-core arithmetic model.

The model (tests/tc_arith.py) is a diagnostic description of the kernels'
accumulation, so it has to describe them: on crafted inputs the GEMM must give
the model's value exactly; on random inputs most elements agree bit for bit and
the error norms agree closely."""

import pytest
import torch

from tests import tc_arith
from tests.helpers import library, require_gpu

pytestmark = pytest.mark.gpu

U = 2.0 ** -23
CRAFTED = [
    [(0, 1.0), (1, 0.75 * U)],
    [(0, -1.0), (1, -0.75 * U)],
    [(0, 1.0), (8, 0.75 * U)],
    [(0, 1.0), (1, -1.25 * 2 ** -24)],
    [(0, 1.0), (8, -1.25 * 2 ** -24)],
    [(0, 1.0)] + [(k, 2.0 ** -25) for k in range(1, 5)],
    [(0, 1.0)] + [(k, 2.0 ** -26) for k in range(1, 8)],
    [(0, 1024.0), (1, -1024.0), (2, 3 * 2.0 ** -20)],
    [(0, 1024.0), (8, -1024.0), (9, 3 * 2.0 ** -20)],
    [(0, 1.0), (72, 2.0 ** -24), (100, -3 * 2.0 ** -25)],
]


@pytest.mark.parametrize("prec", ["tf32", "3xtf32"])
@pytest.mark.parametrize("dim", [128, 256])
def test_crafted_inputs_follow_the_rule(prec, dim):
    require_gpu()
    dr = library()
    n = len(CRAFTED)
    A = torch.zeros((n, dim, dim), device="cuda")
    B = torch.zeros((n, dim, dim), device="cuda")
    for z, terms in enumerate(CRAFTED):
        for k, v in terms:
            A[z, 0, k] = v
            B[z, k, 0] = 1.0
    kw = dict(A_lo=torch.zeros_like(A), B_lo=torch.zeros_like(B)) if prec == "3xtf32" else {}
    C = dr.gemm(A, B, prec=prec, **kw)
    sub = tc_arith.partial_sub_for(dim, prec)
    for z in range(n):
        want = tc_arith.gemm(A[z, :1], B[z, :, :1], prec, sub)[0, 0]
        assert float(C[z, 0, 0]) == float(want), (z, float(C[z, 0, 0]), float(want))


@pytest.mark.parametrize("prec", ["tf32", "3xtf32"])
@pytest.mark.parametrize("dim", [128, 256, 1024])
def test_random_products_track_the_model(prec, dim):
    require_gpu()
    dr = library()
    g = torch.Generator(device="cuda").manual_seed(dim)
    A = torch.randn((1, dim, dim), device="cuda", generator=g)
    A = A * torch.exp(torch.randn((1, dim, dim), device="cuda", generator=g))
    B = torch.randn((1, dim, dim), device="cuda", generator=g)
    if prec == "3xtf32":
        ah, al = tc_arith.split_tf32(A)
        bh, bl = tc_arith.split_tf32(B)
        C = dr.gemm(ah, bh, prec="3xtf32", A_lo=al, B_lo=bl)[0]
        ex = (ah + al)[0].double() @ (bh + bl)[0].double()
    else:
        ah, bh = tc_arith.rna_tf32(A), tc_arith.rna_tf32(B)
        C = dr.gemm(ah, bh, prec="tf32")[0]
        ex = ah[0].double() @ bh[0].double()
    rows = min(dim, 256)
    M = tc_arith.gemm(A[0, :rows], B[0], prec, tc_arith.partial_sub_for(dim, prec))
    same = (M == C[:rows]).double().mean().item()
    eg = ((C[:rows].double() - ex[:rows]).norm() / ex[:rows].norm()).item()
    em = ((M.double() - ex[:rows]).norm() / ex[:rows].norm()).item()
    print("dim %d %s: identical %.3f, error gpu %.3e model %.3e" % (dim, prec, same, eg, em))
    assert same > 0.7
    assert abs(eg - em) < 0.05 * em
