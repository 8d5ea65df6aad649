"""GPU path against the float64 oracle on the same seeded inputs.

Each test hands the oracle the exact fp32 bits the GPU consumed (and, for the
root solvers, the GPU's own fp32 scale), so every step is checked on its own.
Gates (relative Frobenius error of the result, per block):
  3xTF32 1e-4, TF32 2e-3, FP16/BF16 Coupled Newton and Chebyshev 1e-2;
  NDB in half precision is reported, not gated (the pages call it unstable).
Power-iteration lambda: relative error 1e-5 (3xTF32 products); the half-precision
modes are checked against the oracle run on the same 16-bit A (see
test_power_lambda_half).  Accumulate / apply: 1e-5 / 1e-4.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import library, rel_fro_blocks, require_gpu, rna_tf32, to64

pytestmark = pytest.mark.gpu

GATE = {"3xtf32": 1e-4, "tf32": 2e-3, "fp16": 1e-2, "bf16": 1e-2}
PRECS = ["3xtf32", "tf32", "fp16", "bf16"]


def wishart_case(n, b, seed):
    A = synth.wishart(n, b, seed=seed, device="cuda")
    V0 = synth.start_vectors(n, b, 32, seed=seed + 1, device="cuda")
    return A, V0


@pytest.mark.parametrize("b", [128, 384])
def test_power_lambda(b):
    require_gpu()
    dr = library()
    A, V0 = wishart_case(8, b, 1000 + b)
    for iters, nv in ((10, 32), (1, 5), (3, 17)):
        lam = dr.spectral_scale(A, dr.SCALE_POWER, V0[:, :, :nv].contiguous(), iters, ridge=1e-3)
        torch.cuda.synchronize()
        ref = oracle.power_lambda(to64(A), to64(V0[:, :, :nv]), iters, ridge=1e-3)
        assert np.max(np.abs(to64(lam) - ref) / ref) < 1e-5, (iters, nv)
    assert dr.device_status() == 0


HALF_MODES = [("fp16", torch.float16, 2.0 ** -11), ("bf16", torch.bfloat16, 2.0 ** -8)]


@pytest.mark.parametrize("name,dt,u", HALF_MODES)
@pytest.mark.parametrize("b,n", [(128, 8), (256, 200), (384, 9), (1024, 4), (1024, 40), (2048, 2)])
def test_power_lambda_half(name, dt, u, b, n):
    """Half-precision power iteration ([pt] Principais Contribuicoes item 4).

    Against the oracle on the 16-bit A the GPU read, the differences are the
    16-bit rounding of the vectors between products (relative u) and fp32 sums.
    A perturbation dv of the final vector changes its Rayleigh quotient by at most
    2 |dv| |(A - rho I) v| / |v|^2 <= 2u ||A||_2, so the gate is 4u.  The ridge,
    0.2 here (about 7% of lambda), is large enough that dropping it fails that
    gate in both formats.  Against the oracle on the fp32 A, the 16-bit rounding E
    of A (|E_ij| <= u |A_ij|) moves every eigenvalue by at most
    ||E||_2 <= u ||A||_F (Weyl), which bounds that difference."""
    require_gpu()
    dr = library()
    mode = dr.SCALE_POWER_F16 if name == "fp16" else dr.SCALE_POWER_BF16
    A, V0 = wishart_case(n, b, 1900 + b)
    for iters, nv in ((10, 32), (3, 7)):
        V = V0[:, :, :nv].contiguous()
        lam = to64(dr.spectral_scale(A, mode, V, iters, ridge=0.2))
        sig = half_power_sigma(A, 0.2)
        Ah = to64((A * sig[:, None, None]).to(dt)) / to64(sig)[:, None, None]
        ref_h = oracle.power_lambda(Ah, to64(V), iters, ridge=0.2)
        err_h = np.abs(lam - ref_h) / ref_h
        print("%s B=%d iters=%d nv=%d: vs oracle on the 16-bit A %.2e" % (
            name, b, iters, nv, err_h.max()))
        assert err_h.max() < 4 * u, (iters, nv, err_h)
        ref = oracle.power_lambda(to64(A), to64(V), iters, ridge=0.2)
        bound = u * np.linalg.norm(to64(A).reshape(n, -1), axis=1) / ref
        assert np.all(np.abs(lam - ref) / ref <= bound + 4 * u)
    assert dr.device_status() == 0


@pytest.mark.parametrize("name,dt,u", HALF_MODES)
@pytest.mark.parametrize("b,n,iters,nv", [
    (1024, 1, 1, 1),      # one block: one cluster, lane 1 empty, a single product
    (128, 1, 2, 32),      # clusters of one CTA
    (640, 7, 1, 3),       # clusters of 5 CTAs, lanes without a stagger (one product)
    (896, 3, 4, 16),      # clusters of 7 CTAs, an odd block count
    (128, 1000, 10, 32),  # many blocks per cluster: every scratch slot reused
    (256, 700, 3, 32),
    (1024, 64, 10, 32),   # blocks of 1024, four or five per cluster
])
def test_power_lambda_half_shapes(name, dt, u, b, n, iters, nv):
    """The half-precision iteration over block orders, counts and iteration counts
    that exercise its launch shapes (cluster size B / 128, blocks per cluster, the
    lanes' start offset, the slots' reuse).  Gate: 4u against the oracle on the
    16-bit A, as in test_power_lambda_half."""
    require_gpu()
    dr = library()
    mode = dr.SCALE_POWER_F16 if name == "fp16" else dr.SCALE_POWER_BF16
    A, V0 = wishart_case(n, b, 2300 + b + n)
    V = V0[:, :, :nv].contiguous()
    lam = to64(dr.spectral_scale(A, mode, V, iters, ridge=0.2))
    sig = half_power_sigma(A, 0.2)
    Ah = to64((A * sig[:, None, None]).to(dt)) / to64(sig)[:, None, None]
    ref_h = oracle.power_lambda(Ah, to64(V), iters, ridge=0.2)
    err_h = np.abs(lam - ref_h) / ref_h
    print("%s B=%d N=%d iters=%d nv=%d: vs oracle on the 16-bit A %.2e" % (
        name, b, n, iters, nv, err_h.max()))
    assert err_h.max() < 4 * u, err_h
    assert dr.device_status() == 0


def half_power_sigma(A, ridge):
    """The exact power of two the half modes scale each block by, as the header
    states it: 2^-e with max(max_i |A_ii|, |ridge|) = f 2^e, f in [1/2, 1)."""
    m = np.maximum(np.abs(np.diagonal(to64(A), axis1=1, axis2=2)).max(axis=1), abs(ridge))
    _, e = np.frexp(m)
    e = np.clip(e, -126, 126)
    return torch.tensor(np.ldexp(1.0, -e), dtype=torch.float32, device=A.device)


@pytest.mark.parametrize("name,dt,u", HALF_MODES)
def test_power_half_scale_invariant(name, dt, u):
    """The half modes store sigma A with sigma an exact power of two, so the 16-bit
    copy of 2^k A (ridge 2^k r) is bit for bit that of A, and lambda scales by 2^k
    up to the order of the fp32 column-sum atomics.  At k = -40 an unscaled fp16
    copy of A would be all zeros (lambda = the ridge alone) and at k = 20 it would
    overflow to inf, so each scaled run is checked against the oracle at its own
    scale with the bound of test_power_lambda_half."""
    require_gpu()
    dr = library()
    mode = dr.SCALE_POWER_F16 if name == "fp16" else dr.SCALE_POWER_BF16
    A, V0 = wishart_case(4, 256, 2200)
    ref0 = oracle.power_lambda(to64(A), to64(V0), 10, ridge=0.2)
    bound = u * np.linalg.norm(to64(A).reshape(4, -1), axis=1) / ref0 + 4 * u
    lam0 = to64(dr.spectral_scale(A, mode, V0, 10, ridge=0.2))
    for k in (0, -40, -20, 20):
        Ak = A * 2.0 ** k
        if k == -40:
            assert torch.count_nonzero(Ak.half()) == 0
        if k == 20:
            assert not torch.isfinite(Ak.half()).all()
        lam = to64(dr.spectral_scale(Ak, mode, V0, 10, ridge=0.2 * 2.0 ** k))
        ref = ref0 * 2.0 ** k
        err = np.abs(lam - ref) / ref
        print("%s k=%d: vs oracle %.2e, vs k=0 run %.2e" % (
            name, k, err.max(), np.max(np.abs(lam / 2.0 ** k - lam0) / lam0)))
        assert np.all(err <= bound), (k, err, bound)
    assert dr.device_status() == 0


def test_frobenius_scale():
    require_gpu()
    dr = library()
    A, _ = wishart_case(5, 256, 7)
    s = dr.spectral_scale(A, dr.SCALE_FROBENIUS, ridge=0.5)
    ref = oracle.frobenius_norm(to64(A), ridge=0.5)
    assert np.max(np.abs(to64(s) - ref) / ref) < 1e-5


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("iters", [1, 2, 10])
def test_cn_parity(prec, iters):
    require_gpu()
    dr = library()
    A, V0 = wishart_case(8, 128, 1001)
    lam = dr.spectral_scale(A, dr.SCALE_POWER, V0, 10)
    X, r = dr.inv_root_cn(A, lam, iters=iters, prec=prec, resid=True)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    Xr, rr, _ = oracle.cn_inv_root(to64(A), to64(lam), iters)
    err = rel_fro_blocks(to64(X), Xr)
    assert err.max() < GATE[prec], err
    # Residuals are held to the precision's stated root tolerance.
    rerr = np.max(np.abs(to64(r) - rr)) / max(1.0, rr.max())
    print("CN %s iters=%d root err %.3e, residual err %.3e" % (prec, iters, err.max(), rerr))
    assert rerr < GATE[prec]


def rank_deficient_factors(n, b, seed):
    """Factors G G^T (scaled by 1 - beta = 0.05) of bf16 gradient blocks whose right
    half is zero padding: rank b / 2, so with a 1e-6 ridge the scaled condition
    number is about 1e6 -- the padded factors of the Llama workload."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    G = (0.1 * torch.randn((n, b, b), generator=g, device="cuda")).to(torch.bfloat16).float()
    G[:, :, b // 2:] = 0
    return 0.05 * torch.bmm(G, G.transpose(1, 2))


@pytest.mark.parametrize("b", [256, 512, 384])
def test_cn_half_ill_conditioned(b):
    """16-bit Coupled Newton on ill-conditioned factors against the oracle.

    Rounding M to 16 bits moves the smallest scaled eigenvalues (about 1e-6) by
    far more than themselves; the early M-updates therefore read M as a 16-bit
    pair (hi + lo).  FP16 is held to its 1e-2 gate.  BF16's 8-bit iterates X and
    T cannot reach it at this condition number: reported, not gated."""
    require_gpu()
    dr = library()
    ridge = 1e-6
    F = rank_deficient_factors(6, b, 5000 + b)
    V0 = synth.start_vectors(6, b, 32, seed=5100 + b, device="cuda")
    lam = dr.spectral_scale(F, dr.SCALE_POWER, V0, 10, ridge=ridge)
    ref = oracle.cn_inv_root(to64(F), to64(lam), 10, ridge=ridge)[0]
    for prec in ("fp16", "bf16"):
        X = dr.inv_root_cn(F, lam, 10, prec, ridge=ridge)
        torch.cuda.synchronize()
        assert dr.device_status() == 0
        err = rel_fro_blocks(to64(X), ref)
        print("CN %s B=%d rank-deficient factors: max rel err %.3e" % (prec, b, err.max()))
        assert np.all(np.isfinite(to64(X)))
        if prec == "fp16":
            assert err.max() < GATE[prec], err


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("iters", [1, 2, 10])
def test_ndb_parity(prec, iters):
    require_gpu()
    dr = library()
    A, V0 = wishart_case(8, 128, 1002)
    lam = dr.spectral_scale(A, dr.SCALE_POWER, V0, 10)
    X, r = dr.inv_root_ndb(A, lam, iters=iters, prec=prec, resid=True)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    Xr, rr, _ = oracle.ndb_inv_root(to64(A), to64(lam), iters)
    err = rel_fro_blocks(to64(X), Xr)
    rerr = np.max(np.abs(to64(r) - rr)) / max(1.0, rr.max())
    print("NDB %s iters=%d max rel err %.3e, residual err %.3e" % (prec, iters, err.max(), rerr))
    if prec in ("3xtf32", "tf32"):
        # Roots and residuals are held to the precision's stated root tolerance.
        assert err.max() < GATE[prec], err
        assert rerr < GATE[prec], rerr
    else:
        pass  # half-precision NDB: reported above, not gated


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("degree", [1, 2, 3, 16])
def test_cheb_parity(prec, degree):
    require_gpu()
    dr = library()
    A, V0 = wishart_case(8, 128, 1003)
    lam = dr.spectral_scale(A, dr.SCALE_POWER, V0, 10)
    X = dr.inv_root_cheb(A, lam, degree=degree, lo=1e-2, hi=1.05, prec=prec)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    Xr, _ = oracle.cheb_inv_root(to64(A), to64(lam), degree, 1e-2, 1.05)
    err = rel_fro_blocks(to64(X), Xr)
    assert err.max() < GATE[prec], err


@pytest.mark.parametrize("b", [256, 384])
def test_roots_other_sizes(b):
    require_gpu()
    dr = library()
    A, V0 = wishart_case(3, b, 1004 + b)
    lam = dr.spectral_scale(A, dr.SCALE_POWER, V0, 10)
    lam64 = to64(lam)
    X = dr.inv_root_cn(A, lam, iters=8, prec="3xtf32", ridge=1e-4)
    Xr, _, _ = oracle.cn_inv_root(to64(A), lam64, 8, ridge=1e-4)
    assert rel_fro_blocks(to64(X), Xr).max() < 1e-4
    X = dr.inv_root_ndb(A, lam, iters=6, prec="tf32", ridge=1e-4)
    Xr, _, _ = oracle.ndb_inv_root(to64(A), lam64, 6, ridge=1e-4)
    assert rel_fro_blocks(to64(X), Xr).max() < 2e-3
    X = dr.inv_root_cheb(A, lam, degree=8, prec="3xtf32", ridge=1e-4)
    Xr, _ = oracle.cheb_inv_root(to64(A), lam64, 8, 1e-2, 1.05, ridge=1e-4)
    assert rel_fro_blocks(to64(X), Xr).max() < 1e-4
    assert dr.device_status() == 0


def test_chunked_workspace_is_bitwise_identical():
    require_gpu()
    dr = library()
    A, V0 = wishart_case(8, 128, 1005)
    lam = dr.spectral_scale(A, dr.SCALE_POWER, V0, 10)
    for op, fn, kw in ((dr.OP_INV_ROOT_CN, dr.inv_root_cn, {"iters": 5}),
                       (dr.OP_INV_ROOT_NDB, dr.inv_root_ndb, {"iters": 4}),
                       (dr.OP_INV_ROOT_CHEB, dr.inv_root_cheb, {"degree": 6})):
        full = fn(A, lam, prec="tf32", **kw)
        param = kw.get("iters", kw.get("degree"))
        whole = dr.workspace_size(op, 8, 128, dr.TF32, param)
        small = dr.workspace(op, 8, 128, dr.TF32, param, max_bytes=whole // 3)
        part = fn(A, lam, prec="tf32", ws=small, **kw)
        torch.cuda.synchronize()
        assert torch.equal(full, part), op
    assert dr.device_status() == 0


def test_accumulate_bf16_with_padding():
    require_gpu()
    dr = library()
    ng, b = 4, 256
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    G = (0.1 * torch.randn((ng, b, b), generator=g, device="cuda")).to(torch.bfloat16)
    vr = torch.tensor([256, 200, 256, 128], dtype=torch.int32, device="cuda")
    vc = torch.tensor([256, 256, 72, 128], dtype=torch.int32, device="cuda")
    for j in range(ng):
        G[j, int(vr[j]):, :] = 0
        G[j, :, int(vc[j]):] = 0
    F0 = torch.randn((2 * ng, b, b), generator=g, device="cuda")
    F0 = 0.5 * (F0 + F0.transpose(1, 2))
    F = F0.clone()
    dr.shampoo_accumulate(G, F, 0.95, vr, vc)
    torch.cuda.synchronize()
    ref = oracle.accumulate(to64(F0), to64(G), 0.95, vr.tolist(), vc.tolist())
    assert rel_fro_blocks(to64(F), ref).max() < 1e-5
    # Padded part is exactly the identity's.
    Fh = F.cpu()
    assert torch.equal(Fh[1, 200:, 200:], torch.eye(56))
    assert torch.equal(Fh[ng + 2, 72:, :72], torch.zeros(184, 72))
    assert dr.device_status() == 0


@pytest.mark.parametrize("b", [128, 256, 512])
def test_accumulate_fp32_gradients(b):
    require_gpu()
    dr = library()
    ng = 3
    G = torch.randn((ng, b, b), device="cuda")
    F = torch.zeros((2 * ng, b, b), device="cuda")
    dr.shampoo_accumulate(G, F, 0.9)
    dr.shampoo_accumulate(G, F, 0.9)
    torch.cuda.synchronize()
    ref = oracle.accumulate(np.zeros((2 * ng, b, b)), to64(G), 0.9)
    ref = oracle.accumulate(ref, to64(G), 0.9)
    assert rel_fro_blocks(to64(F), ref).max() < 1e-5
    # A 3xTF32 product adds its two cross terms in opposite orders for (i, j) and
    # (j, i), so tiles computed whole are symmetric to rounding only; the lower
    # 256-tiles of the mirrored path are their mirrors' transposes exactly.
    assert torch.allclose(F, F.transpose(1, 2), rtol=1e-6, atol=1e-6 * float(F.abs().max()))
    t = b // 256
    for i in range(t):
        for j in range(i):
            lo = F[:, i * 256:(i + 1) * 256, j * 256:(j + 1) * 256]
            up = F[:, j * 256:(j + 1) * 256, i * 256:(i + 1) * 256]
            assert torch.equal(lo, up.transpose(1, 2)), (i, j)


def test_accumulate_symmetric_tiles_with_padding():
    """For B a multiple of 256 the factors' upper 256-tiles are computed and the
    lower ones mirrored (SYRK-style).  Checked at B = 768 (3 x 3 tiles), with
    padded rows / columns that cut across tile boundaries: oracle parity, exact
    symmetry, and the identity on the padded part, below the diagonal too."""
    require_gpu()
    dr = library()
    ng, b = 3, 768
    g = torch.Generator(device="cuda")
    g.manual_seed(78)
    G = (0.1 * torch.randn((ng, b, b), generator=g, device="cuda")).to(torch.bfloat16)
    vr = torch.tensor([768, 300, 520], dtype=torch.int32, device="cuda")
    vc = torch.tensor([700, 768, 256], dtype=torch.int32, device="cuda")
    for j in range(ng):
        G[j, int(vr[j]):, :] = 0
        G[j, :, int(vc[j]):] = 0
    F0 = torch.randn((2 * ng, b, b), generator=g, device="cuda")
    F0 = 0.5 * (F0 + F0.transpose(1, 2))
    F = F0.clone()
    for _ in range(2):
        dr.shampoo_accumulate(G, F, 0.95, vr, vc)
    torch.cuda.synchronize()
    ref = oracle.accumulate(to64(F0), to64(G), 0.95, vr.tolist(), vc.tolist())
    ref = oracle.accumulate(ref, to64(G), 0.95, vr.tolist(), vc.tolist())
    assert rel_fro_blocks(to64(F), ref).max() < 1e-5
    assert torch.equal(F, F.transpose(1, 2))
    Fh = F.cpu()
    assert torch.equal(Fh[1, 300:, 300:], torch.eye(468))
    assert torch.equal(Fh[1, 300:, :300], torch.zeros(468, 300))
    assert torch.equal(Fh[ng + 2, 256:, 256:], torch.eye(512))
    assert dr.device_status() == 0


@pytest.mark.parametrize("prec", PRECS)
def test_apply_parity(prec):
    require_gpu()
    dr = library()
    ng, b = 3, 256
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    G = torch.randn((ng, b, b), generator=g, device="cuda").to(torch.bfloat16)
    Fr = synth.wishart(2 * ng, b, seed=9, device="cuda") / 2.0
    U = dr.precondition_apply(G, Fr, prec=prec)
    torch.cuda.synchronize()
    ref = oracle.apply_preconditioner(to64(G), to64(Fr))
    err = rel_fro_blocks(to64(U), ref)
    gate = {"3xtf32": 1e-5, "tf32": 2e-3, "fp16": 5e-3, "bf16": 2e-2}[prec]
    assert err.max() < gate, err


@pytest.mark.parametrize("b", [384, 512])
def test_root_tf32_output(b):
    """DASH_ROOT_TF32 rounds X to TF32 on the way out and changes nothing else: X
    is bit for bit the host's round-to-nearest (ties away) TF32 rounding of the
    plain X, also in the tiles a symmetric-half run completes by transposed
    stores (B = 512)."""
    require_gpu()
    dr = library()
    A, V0 = wishart_case(3, b, 3300 + b)
    s = dr.spectral_scale(A, dr.SCALE_POWER, V0, 10, ridge=1e-3)
    runs = [(dr.inv_root_cn, dict(iters=6), p) for p in ("fp16", "3xtf32", "tf32")]
    runs += [(dr.inv_root_ndb, dict(iters=4), "3xtf32"), (dr.inv_root_cn, dict(iters=1), "fp16"),
             (dr.inv_root_cheb, dict(degree=8, lo=0.02, hi=1.05), "fp16"),
             (dr.inv_root_cheb, dict(degree=1, lo=0.02, hi=1.05), "tf32")]
    for fn, kw, prec in runs:
        X = fn(A, s, prec=prec, ridge=1e-3, **kw)
        Xt = fn(A, s, prec=prec + "+root_tf32", ridge=1e-3, **kw)
        torch.cuda.synchronize()
        assert torch.equal(Xt, rna_tf32(X)), (fn.__name__, kw, prec)
    assert dr.device_status() == 0


def test_apply_reads_tf32_roots_as_they_are():
    """precondition_apply / _update with TF32 | DASH_ROOT_TF32 skip the roots'
    conversion pass: on TF32-rounded roots the results are bit for bit those of
    plain TF32, and they meet the TF32 apply gate against the oracle."""
    require_gpu()
    dr = library()
    ng, b = 3, 512
    g = torch.Generator(device="cuda").manual_seed(3400)
    G = torch.randn((ng, b, b), generator=g, device="cuda").to(torch.bfloat16)
    Fr = rna_tf32(synth.wishart(2 * ng, b, seed=3401, device="cuda") / 2.0)
    U = dr.precondition_apply(G, Fr, prec="tf32")
    Ut = dr.precondition_apply(G, Fr, prec="tf32+root_tf32")
    W0 = torch.randn((ng, b, b), generator=g, device="cuda")
    W, Wt = W0.clone(), W0.clone()
    dr.precondition_update(G, Fr, W, 0.01, "tf32")
    dr.precondition_update(G, Fr, Wt, 0.01, "tf32+root_tf32")
    torch.cuda.synchronize()
    assert torch.equal(U, Ut) and torch.equal(W, Wt)
    ref = oracle.apply_preconditioner(to64(G), to64(Fr))
    assert rel_fro_blocks(to64(Ut), ref).max() < 2e-3
    assert dr.device_status() == 0


def test_empty_stack_is_noop():
    require_gpu()
    dr = library()
    A = torch.empty((0, 128, 128), device="cuda")
    s = torch.empty((0,), device="cuda")
    X = dr.inv_root_cn(A, s, iters=3, ws=torch.empty(256, dtype=torch.uint8, device="cuda"))
    assert X.shape == (0, 128, 128)


PACK_CASES = [((2048, 5632), 5632, torch.bfloat16, 1024),   # a Llama MLP weight, ragged last column
              ((300, 200), 256, torch.float32, 128),        # ragged both ways, row-strided view
              ((128, 384), 384, torch.float16, 128),
              ((300, 203), 210, torch.float32, 128)]         # word-by-word path (cols % 4 != 0)


@pytest.mark.parametrize("shape,ld,dt,b", PACK_CASES)
def test_pack_unpack_bit_exact(shape, ld, dt, b):
    """Weight <-> block stack ([pt] Metodologia 1) against the oracle's cut, bit for bit."""
    require_gpu()
    dr = library()
    rows, cols = shape
    g = torch.Generator(device="cuda").manual_seed(rows + cols)
    base = torch.randn((rows, ld), generator=g, device="cuda").to(dt)
    M = base[:, :cols]
    blocks, vr, vc = dr.pack_blocks(M, b)
    ref, rvr, rvc = oracle.pack_blocks(to64(M), b)
    assert torch.equal(blocks.cpu(), torch.from_numpy(ref).to(dt))  # values are exact in dt
    assert vr.cpu().tolist() == list(rvr) and vc.cpu().tolist() == list(rvc)
    sentinel = torch.full((rows, ld), -7.0, dtype=dt, device="cuda")
    dr.unpack_blocks(blocks, rows, cols, out=sentinel[:, :cols])
    assert torch.equal(sentinel[:, :cols], M)
    assert bool((sentinel[:, cols:] == -7.0).all())  # the gap beyond cols is untouched


def test_pack_llama_layer_layout():
    """Packing one layer's seven weights gives the block layout of the Llama cut."""
    require_gpu()
    dr = library()
    vrs, vcs = [], []
    for rows, cols in synth.llama_weight_shapes(1):
        _, vr, vc = dr.pack_blocks(torch.zeros((rows, cols), dtype=torch.bfloat16, device="cuda"),
                                   1024)
        vrs += vr.cpu().tolist()
        vcs += vc.cpu().tolist()
    assert (vrs, vcs) == tuple(map(list, synth.llama_block_layout(1)))


@pytest.mark.parametrize("prec", ["3xtf32", "tf32"])
def test_precondition_update(prec):
    """W <- W - lr U fused into the apply epilogue, against the oracle's weight step."""
    require_gpu()
    dr = library()
    G, vr, vc = synth.llama_layer_blocks(1, seed=2100, var=1e-2, device="cuda")
    G = G[40:48].contiguous()  # includes zero-padded blocks of the MLP weights
    vr, vc = vr[40:48], vc[40:48]
    ng, b = G.shape[0], G.shape[1]
    g = torch.Generator(device="cuda").manual_seed(2101)
    Q = torch.randn((2 * ng, b, b), generator=g, device="cuda") / b ** 0.5
    Froot = Q @ Q.transpose(1, 2) + torch.eye(b, device="cuda")  # SPD stand-ins for the roots
    # Roots of padded factors are the identity on the padded part (accumulate keeps
    # the factors so), which is what leaves the padding of U zero.
    valid = torch.cat([vr, vc]).tolist()
    for k in range(2 * ng):
        v = int(valid[k])
        Froot[k, v:, :] = 0
        Froot[k, :, v:] = 0
        Froot[k, v:, v:] = torch.eye(b - v, device="cuda")
    W0 = torch.randn((ng, b, b), generator=g, device="cuda")
    for j in range(ng):
        W0[j, int(vr[j]):, :] = 0
        W0[j, :, int(vc[j]):] = 0
    W = W0.clone()
    U = torch.empty_like(W)
    lr = 0.01
    dr.precondition_update(G, Froot, W, lr, prec, U=U)
    U_apply = dr.precondition_apply(G, Froot, prec)
    torch.cuda.synchronize()
    assert torch.equal(U, U_apply)  # same products, same epilogue arithmetic
    ref = oracle.update_weights(to64(W0), to64(G), to64(Froot), lr)
    step = to64(W) - to64(W0)
    err = rel_fro_blocks(step, ref - to64(W0))
    print("update %s: step rel err max %.3e" % (prec, err.max()))
    assert err.max() < GATE[prec]
    for j in range(ng):  # padded parts of W stay exactly as they were
        assert bool((W[j, int(vr[j]):, :] == 0).all()) and bool((W[j, :, int(vc[j]):] == 0).all())


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("b", [512, 1024])
def test_symmetric_half_iterates(prec, b):
    """B a multiple of 256: CN and Chebyshev keep symmetric-half iterates (only the
    256-tiles on or above the diagonal are computed).  Chebyshev degrees 3, 4 and 5
    take b_2 from the prologue, the first product and the loop respectively; the
    last product reads it whole."""
    require_gpu()
    dr = library()
    A, _ = wishart_case(3, b, 2200 + b)
    s = dr.spectral_scale(A, dr.SCALE_FROBENIUS)
    X = dr.inv_root_cn(A, s, 8, prec)
    err = rel_fro_blocks(to64(X), oracle.cn_inv_root(to64(A), to64(s), 8)[0])
    assert err.max() < GATE[prec], ("cn", err)
    for d in (3, 4, 5, 8):
        X = dr.inv_root_cheb(A, s, d, 1e-2, 1.05, prec)
        ref = oracle.cheb_inv_root(to64(A), to64(s), d, 1e-2, 1.05)[0]
        err = rel_fro_blocks(to64(X), ref)
        assert err.max() < GATE[prec], ("cheb", d, err)
        assert np.all(np.isfinite(to64(X)))


def test_auto_roots_with_interleaved_tiers():
    """Per-block solver choice ([pt] Significancia e Alegacoes, Direcoes Futuras) on a
    stack whose blocks alternate between the two default tiers, so that each tier is
    gathered into a sub-stack, solved and scattered back.  The choice must be the
    oracle's rule on the GPU's estimates, and every root must meet its tier's gate
    against the oracle (the 3xTF32 tier at most twice a plain float32 run's error
    where that exceeds 1e-4)."""
    require_gpu()
    dr = library()
    n, b = 8, 256
    A = synth.two_cluster_blocks(n, b, 4242, device="cuda")
    V0 = synth.start_vectors(n, b, 32, seed=4243, device="cuda")
    lam = dr.spectral_scale(A, dr.SCALE_POWER, V0, 10)
    lmin = dr.spectral_lambda_min(A, lam, dr.SCALE_POWER, V0, 10)
    tiers = dr.DEFAULT_TIERS
    X, choice = dr.inv_root_auto(A, lam, lmin, tiers)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    lam64, lmin64 = to64(lam), to64(lmin)
    want = oracle.select_tiers(oracle.condition_estimate(lam64, lmin64), tiers)
    assert choice == want.tolist()
    assert choice == [k % 2 for k in range(n)], choice
    A64 = to64(A)
    ref = oracle.auto_inv_root(A64, lam64, np.array(choice), tiers)
    err = rel_fro_blocks(to64(X), ref)
    for k in range(n):
        tier = tiers[choice[k]]
        gate = tier["gate"]
        if tier["prec"] == "3xtf32":
            x32 = oracle.cn_inv_root(A64[k:k + 1], lam64[k:k + 1], tier["iters"],
                                     dtype=np.float32)[0]
            gate = max(gate, 2.0 * rel_fro_blocks(x32, ref[k:k + 1])[0])
        print("auto block %d tier %d: rel err %.3e, gate %.3e" % (k, choice[k], err[k], gate))
        assert err[k] < gate, (k, err[k], gate)
