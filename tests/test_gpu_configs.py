"""The five workload configurations at full size, against the float64 oracle.

Each test runs the GPU path on the whole stack, in the launch configuration
bench.py times, and checks sampled blocks against the oracle run on the exact fp32
inputs (and the GPU's own fp32 scales).  Gates (relative Frobenius error per
block): 3xTF32 1e-4, TF32 2e-3, FP16/BF16 Coupled Newton 1e-2; half-precision
NDB is reported, not gated.  Measured errors are printed (run with -s).

Ill-conditioned stacks.  Configs 2-4 have scaled condition numbers of 1e6-1e7
(a spectrum down to 1e-6, or rank-deficient Gram matrices plus a 1e-6 ridge).
There the inverse 4th root of the smallest eigen-directions is so sensitive that
arithmetic of the path's own precision may miss the stated gate.
  * 3xTF32 / TF32 roots: a sampled block that misses the stated gate is rerun
    with the test-side model of the library's tensor-core arithmetic
    (tests/tc_arith.py: alignment truncation with two guard bits, round toward
    zero, the kernels' partial structure), in float64 on the GPU.  Its gate is
    R_TC times the model's own error, and the GPU root must lie within
    TRACK_TC times that error of the model's root.
  * FP16 / BF16 roots: the root is also computed on the CPU with the library's
    storage rule (iterates rounded to the storage type, products in float32);
    the gate is R_EMUL times that emulation's error when the emulation itself
    misses the stated gate.
Every other stage of those configs (accumulate, lambda, apply, padding) keeps
its stated gate.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import tc_arith
from tests.helpers import (cn_emulated, library, ndb_emulated, rel_fro, rel_fro_blocks,
                           require_gpu, to64)

pytestmark = pytest.mark.gpu

GATE = {"3xtf32": 1e-4, "tf32": 2e-3, "fp16": 1e-2, "bf16": 1e-2}
RIDGE = 1e-6


R_EMUL = 10.0
R_TC = 1.5
TRACK_TC = 0.25
MAX_TC_BLOCKS = 8


def check_root(name, X, A, lam, idx, ref_fn, gate, emul_fn=None, tc_fn=None):
    """Relative Frobenius error of X[idx] against the oracle.

    With tc_fn (3xTF32 / TF32 on ill-conditioned stacks) the blocks that miss the
    stated gate are rerun with the tensor-core arithmetic model (at most
    MAX_TC_BLOCKS of them, the worst first; any others must then stay below the
    largest gate so found).  With emul_fn (half precision) the same iteration is
    run on the CPU in the storage precision; the gate becomes R_EMUL times that
    emulation's error whenever the emulation itself misses the stated gate."""
    Xs = to64(X[idx])
    A64 = to64(A[idx])
    ref = ref_fn(A64, to64(lam[idx]))
    err = rel_fro_blocks(Xs, ref)
    msg = "%s: blocks %s rel err max %.3e" % (name, [int(i) for i in idx], err.max())
    if tc_fn is not None:
        print(msg)
        assert np.all(np.isfinite(Xs))
        miss = [t for t in np.argsort(-err) if err[t] >= gate]
        gates = np.full(len(idx), gate)
        for t in miss[:MAX_TC_BLOCKS]:
            i = int(idx[t])
            xm = to64(tc_fn(A[i], float(lam[i])))
            em = rel_fro(xm, ref[t])
            dm = rel_fro(Xs[t], xm)
            gates[t] = max(gate, R_TC * em)
            print("   block %d: gpu %.3e, tensor-core model %.3e, gpu vs model %.3e"
                  % (i, err[t], em, dm))
            assert dm < TRACK_TC * em, (name, i, dm, em)
        for t in miss[MAX_TC_BLOCKS:]:
            gates[t] = gates.max()
        assert np.all(err < gates), (name, err, gates)
        return err
    if emul_fn is not None:
        xe = np.stack([emul_fn(A[int(i)].cpu(), float(lam[int(i)])) for i in idx])
        ee = rel_fro_blocks(xe, ref)
        g = gate if ee.max() <= gate else R_EMUL * ee.max()
        msg += " (CPU emulation in the same precision: %.3e; gate %.1e)" % (ee.max(), g)
        print(msg)
        assert np.all(np.isfinite(Xs))
        assert err.max() < g, (name, err, ee)
        return err
    print(msg)
    if gate is not None:
        assert err.max() < gate, (name, err)
    return err


def test_config1_small_all_solvers():
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
        check_root("cfg1 CN %s" % prec, X, A, lam, idx,
                   lambda a, s: oracle.cn_inv_root(a, s, 10)[0], GATE[prec])
        print("   CN %s vs EVD %.3e" % (prec, rel_fro_blocks(to64(X), evd).max()))
        X = dr.inv_root_ndb(A, lam, 10, prec)
        check_root("cfg1 NDB %s" % prec, X, A, lam, idx,
                   lambda a, s: oracle.ndb_inv_root(a, s, 10)[0],
                   GATE[prec] if prec in ("3xtf32", "tf32") else None)
        print("   NDB %s vs EVD %.3e" % (prec, rel_fro_blocks(to64(X), evd).max()))
        X = dr.inv_root_cheb(A, lam, 16, 1e-2, 1.05, prec)
        check_root("cfg1 Cheb16 %s" % prec, X, A, lam, idx,
                   lambda a, s: oracle.cheb_inv_root(a, s, 16, 1e-2, 1.05)[0], GATE[prec])
    assert dr.device_status() == 0


def iterations_to(resid, tol):
    """First iteration index whose residual is <= tol (len if never), per row."""
    hit = resid <= tol
    return np.where(hit.any(axis=-1), hit.argmax(axis=-1), resid.shape[-1])


def test_config2_frobenius_vs_power_scaling():
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
        print("cfg2 %s %s: iterations to 1e-3 mean %.1f min %d max %d" % (k + (v.mean(), v.min(), v.max())))
    # Frobenius scaling pushes the spectrum towards zero and needs more iterations.
    assert its[("cn", "power")].mean() < its[("cn", "frobenius")].mean()
    assert its[("ndb", "power")].mean() < its[("ndb", "frobenius")].mean()
    assert its[("cn", "power")].max() < kmax
    # fp32 parity of X at the iteration count the power-scaled CN needed.
    k = int(its[("cn", "power")].max()) + 1
    lam = scales["power"]
    X = dr.inv_root_cn(A, lam, k, "3xtf32")
    check_root("cfg2 CN 3xtf32 K=%d" % k, X, A, lam, np.array([0, 63]),
               lambda a, s: oracle.cn_inv_root(a, s, k)[0], GATE["3xtf32"],
               tc_fn=lambda a, s: tc_arith.cn_root(a, s, k, "3xtf32"))
    kn = int(max(its[("ndb", "power")].max() // 2 + 2, 8))
    X = dr.inv_root_ndb(A, lam, kn, "3xtf32")
    check_root("cfg2 NDB 3xtf32 K=%d" % kn, X, A, lam, np.array([0, 63]),
               lambda a, s: oracle.ndb_inv_root(a, s, kn)[0], GATE["3xtf32"],
               tc_fn=lambda a, s: tc_arith.ndb_root(a, s, kn, "3xtf32"))
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
    ref_fn = ((lambda a, s: oracle.ndb_inv_root(a, s, 10, ridge=RIDGE)[0]) if root == "ndb"
              else (lambda a, s: oracle.cn_inv_root(a, s, 10, ridge=RIDGE)[0]))
    emul = ((lambda a, s: ndb_emulated(a, s, 10, prec, RIDGE)) if root == "ndb"
            else (lambda a, s: cn_emulated(a, s, 10, prec, RIDGE)))
    tc = ((lambda a, s: tc_arith.ndb_root(a, s, 10, prec, RIDGE)) if root == "ndb"
          else (lambda a, s: tc_arith.cn_root(a, s, 10, prec, RIDGE)))
    gate = GATE[prec] if (root == "cn" or prec in ("3xtf32", "tf32")) else None
    name = "%s %s %s" % (tag, root, prec)
    if gate is None:  # half-precision NDB: reported only
        check_root(name, X, F, lam, fidx, ref_fn, None)
    elif prec in ("3xtf32", "tf32"):
        check_root(name, X, F, lam, fidx, ref_fn, gate, tc_fn=tc)
    else:
        check_root(name, X, F, lam, fidx, ref_fn, gate, emul)
    Xs = torch.cat([X[gidx], X[ng + gidx]])
    Uref = oracle.apply_preconditioner(G64, to64(Xs))
    errU = rel_fro_blocks(to64(U[gidx]), Uref)
    print("%s apply rel err max %.3e" % (tag, errU.max()))
    assert errU.max() < (1e-4 if prec == "3xtf32" else 2e-3)
    print("%s sampled factors: scaled lambda_min %s" % (
        tag, ["%.1e" % (np.linalg.eigvalsh(to64(F[int(i)]) + RIDGE * np.eye(1024))[0] / float(lam[int(i)]))
              for i in fidx[:4]]))
    assert dr.device_status() == 0


def test_config3_one_llama_layer_ndb_fp32():
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
    check_step(dr, "cfg3", G, vr, vc, F, V0, lam, X, U, "ndb", "3xtf32", fidx, gidx)
    # The root of a padded factor is close to the identity on the padded part.
    Xp = to64(X[ng + padded[0]])[512:, 512:]
    print("cfg3 padded root deviation from I: %.3e" % np.abs(Xp - np.eye(512)).max())


@pytest.mark.parametrize("root,prec", [("cn", "fp16"), ("ndb", "3xtf32")])
def test_config4_24_layer_step(root, prec):
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
    check_step(dr, "cfg4", *out, root, prec, fidx, gidx, power="fp16")


SWEEP = [(256, 61035, 4), (512, 15259, 3), (1024, 3815, 2), (2048, 954, 1)]


@pytest.mark.parametrize("b,n,nsample", SWEEP)
def test_config5_sweep(b, n, nsample):
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
        check_root("cfg5 B=%d %s %s" % (b, solver, prec), X, A, s, idx, ref_fn, GATE[prec])
    assert dr.device_status() == 0
