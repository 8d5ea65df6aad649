"""The five benchmark workloads at full size, against the float64 oracle: 8 Wishart
blocks of 128; 64 blocks of 512 with a 1e-6 spectrum; one Llama-d2048 layer (NDB
3xTF32); the 24-layer Llama step ((2496, 1024, 1024) factors); Wishart stacks of
about 16 GB at B = 256 ... 2048.

Each test runs the GPU path on the whole stack, in the launch configuration
bench.py times, and checks sampled blocks against the oracle run on the exact fp32
inputs (and the GPU's own fp32 scales).  Gates (relative Frobenius error per
block, against the float64 oracle running the same iteration): 3xTF32 1e-4, TF32
2e-3, FP16/BF16 Coupled Newton 1e-2; half-precision NDB is reported, not gated.
Every block's error and gate are printed (run with -s).

Ill-conditioned stacks.  The spectrum and Llama stacks have scaled condition numbers of 1e6-1e7
(a spectrum down to 1e-6, or rank-deficient Gram matrices plus a 1e-6 ridge).  On
such a block even a plain round-to-nearest float32 run of the same iteration (the
oracle's own steps in float32: oracle.cn_inv_root / ndb_inv_root with
dtype=np.float32) may miss 1e-4.  A 3xTF32 block is then held to F32_FACTOR times
that float32 run's error instead: the fp32-class path must be as accurate as
ordinary float32 arithmetic, within a factor of two.  The float32 run shares
nothing with the kernels (no partial sums, no truncation model, no tile mirroring).
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import library, rel_fro_blocks, require_gpu, to64

pytestmark = pytest.mark.gpu

GATE = {"3xtf32": 1e-4, "tf32": 2e-3, "fp16": 1e-2, "bf16": 1e-2}
RIDGE = 1e-6
F32_FACTOR = 2.0


def check_root(name, X, A, lam, idx, ref_fn, gate, f32_fn=None):
    """Relative Frobenius error of X[idx] against the oracle, per block.

    ref_fn(A64, lam64) is the float64 oracle.  With f32_fn (3xTF32 roots of
    ill-conditioned stacks) -- the same iteration in plain float32 -- a block whose
    float32 run misses the stated gate is held to F32_FACTOR times that run's error.
    gate None: reported only."""
    Xs = to64(X[idx])
    A64 = to64(A[idx])
    l64 = to64(lam[idx])
    ref = ref_fn(A64, l64)
    err = rel_fro_blocks(Xs, ref)
    gates = np.full(len(idx), np.inf if gate is None else gate)
    e32 = None
    if f32_fn is not None and gate is not None:
        e32 = rel_fro_blocks(f32_fn(A64, l64), ref)
        gates = np.maximum(gates, F32_FACTOR * e32)
    for t, i in enumerate(idx):
        print("%s block %d: rel err %.3e, gate %.3e%s" % (
            name, int(i), err[t], gates[t],
            "" if e32 is None else " (float32 run %.3e)" % e32[t]))
    assert np.all(np.isfinite(Xs)), name
    assert np.all(err < gates), (name, err, gates)
    return err


def cn_ref(k, ridge=0.0):
    return lambda a, s: oracle.cn_inv_root(a, s, k, ridge=ridge)[0]


def cn_f32(k, ridge=0.0):
    return lambda a, s: oracle.cn_inv_root(a, s, k, ridge=ridge, dtype=np.float32)[0]


def ndb_ref(k, ridge=0.0):
    return lambda a, s: oracle.ndb_inv_root(a, s, k, ridge=ridge)[0]


def ndb_f32(k, ridge=0.0):
    return lambda a, s: oracle.ndb_inv_root(a, s, k, ridge=ridge, dtype=np.float32)[0]


def test_wishart8_b128_all_solvers():
    """N=8, B=128 Wishart + 1e-6 I: power scale (32 vectors), CN / NDB (10 its), Cheb 16."""
    require_gpu()
    dr = library()
    A = synth.wishart(8, 128, seed=1001, device="cuda")
    V0 = synth.start_vectors(8, 128, 32, seed=2001, device="cuda")
    lam = dr.spectral_scale(A, dr.SCALE_POWER, V0, 10)
    lam_ref = oracle.power_lambda(to64(A), to64(V0), 10)
    assert np.max(np.abs(to64(lam) - lam_ref) / lam_ref) < 1e-5
    evd = oracle.evd_inv_root(to64(A))
    idx = np.arange(8)
    for prec in ("3xtf32", "tf32", "fp16", "bf16"):
        X = dr.inv_root_cn(A, lam, 10, prec)
        check_root("wishart b128 CN %s" % prec, X, A, lam, idx,
                   lambda a, s: oracle.cn_inv_root(a, s, 10)[0], GATE[prec])
        print("   CN %s vs EVD %.3e" % (prec, rel_fro_blocks(to64(X), evd).max()))
        X = dr.inv_root_ndb(A, lam, 10, prec)
        check_root("wishart b128 NDB %s" % prec, X, A, lam, idx,
                   lambda a, s: oracle.ndb_inv_root(a, s, 10)[0],
                   GATE[prec] if prec in ("3xtf32", "tf32") else None)
        print("   NDB %s vs EVD %.3e" % (prec, rel_fro_blocks(to64(X), evd).max()))
        X = dr.inv_root_cheb(A, lam, 16, 1e-2, 1.05, prec)
        check_root("wishart b128 Cheb16 %s" % prec, X, A, lam, idx,
                   lambda a, s: oracle.cheb_inv_root(a, s, 16, 1e-2, 1.05)[0], GATE[prec])
    assert dr.device_status() == 0


def iterations_to(resid, tol):
    """First iteration index whose residual is <= tol (len if never), per row."""
    hit = resid <= tol
    return np.where(hit.any(axis=-1), hit.argmax(axis=-1), resid.shape[-1])


def test_spectrum1e6_b512_power_vs_frobenius_scaling():
    """N=64, B=512, spectrum log-uniform in [1e-6, 1]: iterations to residual 1e-3."""
    require_gpu()
    dr = library()
    A, _, _ = synth.prescribed_spectrum(64, 512, seed=1002, device="cuda")
    V0 = synth.start_vectors(64, 512, 32, seed=2002, device="cuda")
    scales = {"power": dr.spectral_scale(A, dr.SCALE_POWER, V0, 10),
              "frobenius": dr.spectral_scale(A, dr.SCALE_FROBENIUS)}
    kmax = 60
    its = {}
    for name, s in scales.items():
        _, r = dr.inv_root_cn(A, s, kmax, "3xtf32", resid=True)
        its[("cn", name)] = iterations_to(to64(r), 1e-3)
        _, r = dr.inv_root_ndb(A, s, kmax, "3xtf32", resid=True)
        r = to64(r)
        its[("ndb", name)] = iterations_to(r[:, 0], 1e-3) + iterations_to(r[:, 1], 1e-3)
    for k, v in its.items():
        print("spectrum1e6 b512 %s %s: iterations to 1e-3 mean %.1f min %d max %d" % (k + (v.mean(), v.min(), v.max())))
    # Frobenius scaling pushes the spectrum towards zero and needs more iterations.
    assert its[("cn", "power")].mean() < its[("cn", "frobenius")].mean()
    assert its[("ndb", "power")].mean() < its[("ndb", "frobenius")].mean()
    assert its[("cn", "power")].max() < kmax
    # fp32 parity of X at the iteration count the power-scaled CN needed.
    k = int(its[("cn", "power")].max()) + 1
    lam = scales["power"]
    X = dr.inv_root_cn(A, lam, k, "3xtf32")
    check_root("spectrum1e6 b512 CN 3xtf32 K=%d" % k, X, A, lam, np.array([0, 63]), cn_ref(k),
               GATE["3xtf32"], f32_fn=cn_f32(k))
    kn = int(max(its[("ndb", "power")].max() // 2 + 2, 8))
    X = dr.inv_root_ndb(A, lam, kn, "3xtf32")
    check_root("spectrum1e6 b512 NDB 3xtf32 K=%d" % kn, X, A, lam, np.array([0, 63]), ndb_ref(kn),
               GATE["3xtf32"], f32_fn=ndb_f32(kn))
    assert dr.device_status() == 0


def llama_step(dr, layers, root, prec, seed, power="3xtf32"):
    G, vr, vc = synth.llama_layer_blocks(layers, seed=seed, var=1e-2, device="cuda")
    ng = G.shape[0]
    F = torch.zeros((2 * ng, 1024, 1024), device="cuda")
    dr.shampoo_accumulate(G, F, 0.95, vr, vc)
    V0 = synth.start_vectors(2 * ng, 1024, 32, seed=seed + 1, device="cuda")
    mode = {"3xtf32": dr.SCALE_POWER, "fp16": dr.SCALE_POWER_F16}[power]
    lam = dr.spectral_scale(F, mode, V0, 10, ridge=RIDGE)
    ws = dr.workspace(dr.OP_INV_ROOT_NDB if root == "ndb" else dr.OP_INV_ROOT_CN, 2 * ng, 1024,
                      prec, 10, max_bytes=48 << 30)
    fn = dr.inv_root_ndb if root == "ndb" else dr.inv_root_cn
    X = fn(F, lam, 10, prec, ridge=RIDGE, ws=ws)
    del ws
    U = dr.precondition_apply(G, X, "3xtf32" if prec == "3xtf32" else "tf32")
    torch.cuda.synchronize()
    return G, vr, vc, F, V0, lam, X, U


def check_step(dr, tag, G, vr, vc, F, V0, lam, X, U, root, prec, fidx, gidx, power="3xtf32"):
    ng = G.shape[0]
    G64 = to64(G[gidx])
    Fref = oracle.accumulate(np.zeros((2 * len(gidx), 1024, 1024)), G64, 0.95,
                             to64(vr[gidx]), to64(vc[gidx]))
    Fgpu = np.concatenate([to64(F[gidx]), to64(F[ng + gidx])])
    errF = rel_fro_blocks(Fgpu, Fref)
    print("%s accumulate rel err max %.3e" % (tag, errF.max()))
    assert errF.max() < 1e-5
    if power == "fp16":
        # Half-precision power iteration: against the oracle on the fp16 copy of F
        # the GPU read; gate 4u with u = 2^-11 (derived in test_power_lambda_half).
        lam_ref = oracle.power_lambda(to64(F[fidx].half()), to64(V0[fidx]), 10, ridge=RIDGE)
        lgate = 4 * 2.0 ** -11
    else:
        lam_ref = oracle.power_lambda(to64(F[fidx]), to64(V0[fidx]), 10, ridge=RIDGE)
        lgate = 1e-5
    errl = np.abs(to64(lam[fidx]) - lam_ref) / lam_ref
    print("%s lambda (%s power) rel err max %.3e" % (tag, power, errl.max()))
    assert errl.max() < lgate
    ref_fn = ndb_ref(10, RIDGE) if root == "ndb" else cn_ref(10, RIDGE)
    f32 = ndb_f32(10, RIDGE) if root == "ndb" else cn_f32(10, RIDGE)
    # Half-precision NDB is reported only (the pages report it unstable).
    gate = GATE[prec] if (root == "cn" or prec in ("3xtf32", "tf32")) else None
    name = "%s %s %s" % (tag, root, prec)
    check_root(name, X, F, lam, fidx, ref_fn, gate,
               f32_fn=f32 if prec == "3xtf32" else None)
    Xs = torch.cat([X[gidx], X[ng + gidx]])
    Uref = oracle.apply_preconditioner(G64, to64(Xs))
    errU = rel_fro_blocks(to64(U[gidx]), Uref)
    print("%s apply rel err max %.3e" % (tag, errU.max()))
    assert errU.max() < (1e-4 if prec == "3xtf32" else 2e-3)
    print("%s sampled factors: scaled lambda_min %s" % (
        tag, ["%.1e" % (np.linalg.eigvalsh(to64(F[int(i)]) + RIDGE * np.eye(1024))[0] / float(lam[int(i)]))
              for i in fidx[:4]]))
    assert dr.device_status() == 0


def test_llama_layer_d2048_ndb_3xtf32():
    """One d=2048 layer: 52 bf16 gradient blocks, 104 factors; NDB in fp32 (3xTF32)."""
    require_gpu()
    dr = library()
    out = llama_step(dr, 1, "ndb", "3xtf32", seed=1003)
    G, vr, vc, F, V0, lam, X, U = out
    ng = G.shape[0]
    assert ng == 52
    # Whole-stack accumulate parity; padded R factors hold the identity there.
    Fref = oracle.accumulate(np.zeros((104, 1024, 1024)), to64(G), 0.95, to64(vr), to64(vc))
    assert rel_fro_blocks(to64(F), Fref).max() < 1e-5
    padded = [j for j in range(ng) if int(vc[j]) < 1024]
    assert len(padded) == 6
    Fp = F[ng + padded[0]].cpu()
    assert torch.equal(Fp[512:, 512:], torch.eye(512))
    fidx = np.array([0, 17, ng + 5, ng + padded[0], 2 * ng - 1])
    gidx = np.array([0, padded[0], ng - 1])
    check_step(dr, "llama layer", G, vr, vc, F, V0, lam, X, U, "ndb", "3xtf32", fidx, gidx)
    # The root of a padded factor is close to the identity on the padded part.
    Xp = to64(X[ng + padded[0]])[512:, 512:]
    print("llama layer padded root deviation from I: %.3e" % np.abs(Xp - np.eye(512)).max())


@pytest.mark.parametrize("root,prec", [("cn", "fp16"), ("ndb", "3xtf32")])
def test_llama24_step(root, prec):
    """24 layers: (2496, 1024, 1024) factor stack, the full f=1 step; 16 sampled factors.
    Scaling by the half-precision power iteration, as bench.py runs this step."""
    require_gpu()
    dr = library()
    out = llama_step(dr, 24, root, prec, seed=1004, power="fp16")
    G = out[0]
    ng = G.shape[0]
    assert ng == 1248
    rng = np.random.default_rng(4)
    fidx = np.sort(rng.choice(2 * ng, 16, replace=False))
    gidx = np.sort(rng.choice(ng, 4, replace=False))
    check_step(dr, "llama24", *out, root, prec, fidx, gidx, power="fp16")


def test_llama24_tiered_roots():
    """24 layers, roots with the solver chosen per block ([pt] Significancia e
    Alegacoes, Direcoes Futuras): lambda_min estimates, tier choice and each sampled
    block's root against oracle.lambda_min_estimate / select_tiers / auto_inv_root."""
    require_gpu()
    dr = library()
    G, vr, vc = synth.llama_layer_blocks(24, seed=1004, var=1e-2, device="cuda")
    ng = G.shape[0]
    F = torch.zeros((2 * ng, 1024, 1024), device="cuda")
    dr.shampoo_accumulate(G, F, 0.95, vr, vc)
    del G
    V0 = synth.start_vectors(2 * ng, 1024, 32, seed=1005, device="cuda")
    lam = dr.spectral_scale(F, dr.SCALE_POWER_F16, V0, 10, ridge=RIDGE)
    # The lambda_min iteration in the fp32-accurate mode, so that it has an exact
    # oracle counterpart.
    lmin = dr.spectral_lambda_min(F, lam, dr.SCALE_POWER, V0, 10, ridge=RIDGE)
    TIERS = dr.DEFAULT_TIERS
    X, choice = dr.inv_root_auto(F, lam, lmin, TIERS, ridge=RIDGE, max_ws_bytes=64 << 30)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    lam64, lmin64 = to64(lam), to64(lmin)
    # The tier rule on every block, against the oracle's rule on the same estimates.
    want = oracle.select_tiers(oracle.condition_estimate(lam64, lmin64), TIERS)
    assert choice == want.tolist()
    counts = np.bincount(np.array(choice), minlength=len(TIERS))
    print("llama24 tiers: %s blocks per tier" % counts.tolist())
    # Sample both tiers: 10 random factors plus the first 3 of each tier.
    rng = np.random.default_rng(44)
    fidx = set(rng.choice(2 * ng, 10, replace=False).tolist())
    for t in range(len(TIERS)):
        fidx.update([i for i in range(2 * ng) if choice[i] == t][:3])
    fidx = np.array(sorted(fidx))
    # lambda_min: the oracle's shifted iteration on the same fp32 blocks, start vectors
    # and lambda_max; its eigenvalue estimate mu = lam - lmin to 1e-5 of lam.
    want_min = oracle.lambda_min_estimate(to64(F[fidx]), lam64[fidx], to64(V0[fidx]), 10,
                                          ridge=RIDGE)
    dmin = np.abs(lmin64[fidx] - want_min) / lam64[fidx]
    print("llama24 lambda_min: max |diff| / lambda_max %.3e" % dmin.max())
    assert dmin.max() < 1e-5
    A64 = to64(F[fidx])
    ref = oracle.auto_inv_root(A64, lam64[fidx], np.array(choice)[fidx], TIERS, ridge=RIDGE)
    err = rel_fro_blocks(to64(X[fidx]), ref)
    for t, i in enumerate(fidx):
        tier = TIERS[choice[i]]
        gate = tier["gate"]
        note = ""
        if tier["prec"] == "3xtf32":
            x32 = oracle.cn_inv_root(A64[t:t + 1], lam64[i:i + 1], tier["iters"], ridge=RIDGE,
                                     dtype=np.float32)[0]
            e32 = rel_fro_blocks(x32, ref[t:t + 1])[0]
            gate = max(gate, F32_FACTOR * e32)
            note = " (float32 run %.3e)" % e32
        print("llama24 tiered block %d (tier %d, kappa_hat %.1e): rel err %.3e, gate %.3e%s" % (
            i, choice[i], lam64[i] / max(lmin64[i], 1e-30), err[t], gate, note))
        assert err[t] < gate, (i, err[t], gate)


SWEEP = [(256, 61035, 4), (512, 15259, 3), (1024, 3815, 2), (2048, 954, 1)]


@pytest.mark.parametrize("b,n,nsample", SWEEP)
def test_wishart_sweep_b256_2048(b, n, nsample):
    """Wishart stacks of ~16 GB per B: CN fp16/bf16/tf32/3xtf32, NDB tf32/3xtf32, Cheb 8/16/32."""
    require_gpu()
    dr = library()
    A = synth.wishart(n, b, seed=1005 + b, device="cuda", chunk=256)
    s = dr.spectral_scale(A, dr.SCALE_FROBENIUS)
    V0 = synth.start_vectors(n, b, 32, seed=2005, device="cuda") if n * b * 128 < (8 << 30) else None
    if V0 is not None:
        s = dr.spectral_scale(A, dr.SCALE_POWER, V0, 10)
        del V0
    rng = np.random.default_rng(b)
    idx = np.sort(rng.choice(n, nsample, replace=False))
    X = torch.empty_like(A)
    runs = [("cn", p) for p in ("fp16", "bf16", "tf32", "3xtf32")]
    runs += [("ndb", p) for p in ("tf32", "3xtf32")]
    runs += [("cheb%d" % d, "3xtf32") for d in (8, 16, 32)]
    for solver, prec in runs:
        if solver == "cn":
            ws = dr.workspace(dr.OP_INV_ROOT_CN, n, b, prec, 10, max_bytes=48 << 30)
            dr.inv_root_cn(A, s, 10, prec, X=X, ws=ws)
            ref_fn = lambda a, sc: oracle.cn_inv_root(a, sc, 10)[0]
        elif solver == "ndb":
            ws = dr.workspace(dr.OP_INV_ROOT_NDB, n, b, prec, 10, max_bytes=48 << 30)
            dr.inv_root_ndb(A, s, 10, prec, X=X, ws=ws)
            ref_fn = lambda a, sc: oracle.ndb_inv_root(a, sc, 10)[0]
        else:
            d = int(solver[4:])
            ws = dr.workspace(dr.OP_INV_ROOT_CHEB, n, b, prec, d, max_bytes=48 << 30)
            dr.inv_root_cheb(A, s, d, 1e-2, 1.05, prec, X=X, ws=ws)
            ref_fn = lambda a, sc, d=d: oracle.cheb_inv_root(a, sc, d, 1e-2, 1.05)[0]
        torch.cuda.synchronize()
        del ws
        check_root("sweep B=%d %s %s" % (b, solver, prec), X, A, s, idx, ref_fn, GATE[prec])
    assert dr.device_status() == 0
