"""The tensor-core GEMM engine against float64 products of the same operands.

Covers every operand precision, all four transpose combinations (K-major and
MN-major shared-memory operands), the 128- and 256-wide tile paths and a ragged
multi-tile size (B = 384: three M tiles, three 128-wide N tiles, twelve TF32
k-blocks)."""

import numpy as np
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


def test_graph_replay_and_back_to_back_launches():
    """The mirrored-store pair products (the accumulate, the roots' fp32 results)
    hand out their tiles from a tagged counter at run time.  A launch captured in a
    CUDA graph keeps its tag, so each replay must find the counter cleared by the
    previous run; launches in between take other counters.  Replays of a captured
    accumulate must give the bits of the same accumulates run eagerly."""
    require_gpu()
    dr = library()
    ng, b = 64, 512  # 192 upper pair tiles per launch: more than the pairs, so most come from the counter
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    G = (0.1 * torch.randn((ng, b, b), generator=g, device="cuda")).to(torch.bfloat16)
    F0 = torch.zeros((2 * ng, b, b), device="cuda")
    ref = F0.clone()
    refs = []
    for _ in range(3):
        dr.shampoo_accumulate(G, ref, 0.9)  # eager; also fills the library's caches
        refs.append(ref.clone())
    torch.cuda.synchronize()
    F = F0.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dr.shampoo_accumulate(G, F, 0.9)
    F.copy_(F0)
    for rep in range(3):
        graph.replay()
        for _ in range(rep):
            dr.shampoo_accumulate(G, F0.clone(), 0.9)  # other launches between replays
        torch.cuda.synchronize()
        assert torch.equal(F, refs[rep]), rep
    assert dr.device_status() == 0


def sym_operand(b, n, seed):
    """(n, b, b) fp32 symmetric matrices whose 256-tiles below the diagonal are NaN:
    a symmetric-half product must never read them."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    S = torch.randn((n, b, b), generator=g, device="cuda") / b ** 0.5
    S = 0.5 * (S + S.transpose(1, 2))
    P = S.clone()
    t = b // 256
    for i in range(t):
        for j in range(i):
            P[:, i * 256:(i + 1) * 256, j * 256:(j + 1) * 256] = float("nan")
    return S, P


def upper_tiles(x, b):
    """Mask of the 256-tiles on or above the diagonal."""
    t = b // 256
    m = torch.zeros((b, b), dtype=torch.bool)
    for i in range(t):
        m[i * 256:(i + 1) * 256, i * 256:] = True
    return m.numpy()


@pytest.mark.parametrize("prec", ["tf32", "3xtf32", "fp16", "bf16"])
@pytest.mark.parametrize("sym", [1, 2, 3, 4])
@pytest.mark.parametrize("b", [256, 512, 1024])
def test_gemm_symmetric_halves(prec, sym, b):
    """C = S S, each operand that the mode reads from its upper 256-tiles given
    with NaN below them (A in modes 1, 2, 4; B in 1, 2); modes 2 and 3 write only
    C's upper tiles (C is prefilled with NaN to show what was written)."""
    require_gpu()
    dr = library()
    n = 3
    S, P = sym_operand(b, n, 7 * b + sym)
    Ph, Pl, _ = operands(P, prec)
    Sh, Sl, S64 = operands(S, prec)
    Ah, Al = (Ph, Pl) if sym in (1, 2, 4) else (Sh, Sl)
    Bh, Bl = (Ph, Pl) if sym in (1, 2) else (Sh, Sl)
    C = torch.full((n, b, b), float("nan"), device="cuda")
    dr.gemm_ex(Ah, Bh, prec=prec, sym=sym, A_lo=Al, B_lo=Bl, C=C)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    ref = S64 @ S64
    got = to64(C)
    mask = upper_tiles(got[0], b) if sym in (2, 3) else np.ones((b, b), dtype=bool)
    assert np.all(np.isfinite(got[:, mask]))
    err = np.linalg.norm((got - ref)[:, mask]) / np.linalg.norm(ref[:, mask])
    tol = 2e-5 if prec == "3xtf32" else 1e-5
    assert err < tol, (prec, sym, b, err)


@pytest.mark.parametrize("prec", ["fp16", "bf16"])
@pytest.mark.parametrize("sym", [0, 1, 2])
@pytest.mark.parametrize("b", [128, 256, 384, 512, 1024])
def test_gemm_pair_b(prec, sym, b):
    """16-bit A times a 16-bit pair B = hi + lo: C = A hi + A lo (the product Coupled
    Newton uses for its M iterate), against float64 on the pair's exact value."""
    require_gpu()
    dr = library()
    if sym and b % 256:
        pytest.skip("symmetric halves need B a multiple of 256")
    n = 3
    dt = torch.float16 if prec == "fp16" else torch.bfloat16
    S, P = sym_operand(b, n, 11 * b + sym) if b % 256 == 0 else (None, None)
    if sym == 0 and S is not None:
        P = S  # read whole: no NaN tiles
    if S is None:
        g = torch.Generator(device="cuda")
        g.manual_seed(b)
        S = torch.randn((n, b, b), generator=g, device="cuda") / b ** 0.5
        P = S
    # A = S^2 / 2 commutes with S, so A S is symmetric as sym 2 requires.
    A = (torch.bmm(S, S) * 0.5).to(dt)
    A64 = to64(A)
    if sym:
        A = A.clone()
        for i in range(b // 256):
            for j in range(i):
                A[:, i * 256:(i + 1) * 256, j * 256:(j + 1) * 256] = float("nan")
    hi = P.to(dt)
    lo = (P - hi.float()).to(dt)
    val = to64(S.to(dt)) + to64((S - S.to(dt).float()).to(dt))
    C = torch.zeros((n, b, b), device="cuda")
    dr.gemm_ex(A, hi, prec=prec, sym=sym, B_lo=lo, C=C)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    ref = A64 @ val
    got = to64(C)
    mask = upper_tiles(got[0], b) if sym == 2 else np.ones((b, b), dtype=bool)
    assert np.all(np.isfinite(got[:, mask]))
    err = np.linalg.norm((got - ref)[:, mask]) / np.linalg.norm(ref[:, mask])
    # The lo part must count: without it the error would be the 16-bit rounding of B.
    plain = np.linalg.norm((A64 @ to64(S.to(dt)) - ref)[:, mask]) / np.linalg.norm(ref[:, mask])
    print("pair-B %s sym %d B=%d: rel err %.3e (hi alone %.3e)" % (prec, sym, b, err, plain))
    assert err < 1e-5 and err < 0.05 * plain, (prec, sym, b, err, plain)
