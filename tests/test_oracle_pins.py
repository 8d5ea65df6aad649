"""Pins for the float64 oracle: each check is independent of the oracle's own code.

Every oracle function is tied here to something other than itself: a closed
form, an invariant, a library routine that reaches the same quantity by a
different algorithm, a scalar recurrence written out in plain Python floats, or
brute-force loops on tiny inputs.  A plausible slip in the oracle (a wrong
constant in an iteration, a transposed operand, a dropped term, min for max)
fails at least one of them; ``test_planted_mistakes`` checks that claim for a
few such slips by patching them into copies of the oracle's formulas.
"""

import math

import numpy as np
import numpy.polynomial.chebyshev as npcheb
import pytest
import scipy.linalg

import oracle
import synth


def rel_fro(x, y):
    return float(np.linalg.norm(x - y) / np.linalg.norm(y))


def sym_from_spectrum(lam, seed):
    rng = np.random.default_rng(seed)
    b = len(lam)
    q, r = np.linalg.qr(rng.standard_normal((b, b)))
    q = q * np.sign(np.diag(r))
    return (q * lam) @ q.T, q


# ----------------------------------------------------------------------------- EVD


def test_evd_diagonal_closed_form():
    lam = np.array([1e-4, 0.3, 1.0, 7.0, 1e3])
    X = oracle.evd_inv_root(np.diag(lam)[None])
    np.testing.assert_allclose(X[0], np.diag(lam ** -0.25), rtol=1e-14, atol=1e-15)


def test_evd_two_by_two_by_hand():
    # [[2,1],[1,2]] has eigenpairs 3:(1,1)/sqrt2 and 1:(1,-1)/sqrt2.
    a = np.array([[2.0, 1.0], [1.0, 2.0]])
    r = 3.0 ** -0.25
    want = np.array([[(r + 1) / 2, (r - 1) / 2], [(r - 1) / 2, (r + 1) / 2]])
    np.testing.assert_allclose(oracle.evd_inv_root(a[None])[0], want, rtol=1e-14)


def test_evd_prescribed_spectrum_closed_form():
    A, Q, lam = synth.prescribed_spectrum(3, 48, seed=11, lo=1e-3, hi=1.0)
    A64 = (Q * lam[None, None, :]) @ Q.transpose(1, 2)
    A64 = A64.numpy()
    Q = Q.numpy()
    lam = lam.numpy()
    X = oracle.evd_inv_root(A64)
    for k in range(3):
        want = (Q[k] * lam ** -0.25) @ Q[k].T
        assert rel_fro(X[k], want) < 1e-10


def test_evd_residual_invariant_and_scipy():
    A = synth.wishart(4, 64, seed=3).double().numpy()
    X = oracle.evd_inv_root(A)
    for k in range(4):
        x4 = np.linalg.matrix_power(X[k], 4)
        res = np.linalg.norm(x4 @ A[k] - np.eye(64)) / 8.0
        assert res <= 1e-8
        # Schur-Pade fractional power: a different algorithm for the same function.
        ref = np.real(scipy.linalg.fractional_matrix_power(A[k], -0.25))
        assert rel_fro(X[k], ref) < 1e-9


def test_evd_ridge_and_not_pd():
    A = synth.wishart(2, 16, seed=5, ridge=0.0).double().numpy()
    r = 0.25
    np.testing.assert_allclose(oracle.evd_inv_root(A, ridge=r),
                               oracle.evd_inv_root(A + r * np.eye(16)), rtol=1e-12)
    with pytest.raises(ValueError):
        oracle.evd_inv_root(-np.eye(3)[None])


# ------------------------------------------------------------------- scalar recurrences


def cn_scalar(lam, s, iters, ridge=0.0):
    """Coupled Newton p=4 on one eigenvalue, in plain Python floats."""
    m = (lam + ridge) / s
    x = 1.0
    ms = []
    for _ in range(iters):
        ms.append(m)
        t = (5.0 - m) / 4.0
        x = x * t
        m = m * t ** 4
    return x * s ** -0.25, ms


def ndb_scalar(lam, s, iters, ridge=0.0):
    """Two Newton-Schulz Denman-Beavers stages on one eigenvalue, plain floats."""
    c = (lam + ridge) / s
    qs = []
    y, z = c, 1.0
    for _ in range(iters):
        qs.append(z * y)
        t = (3.0 - z * y) / 2.0
        y, z = y * t, t * z
    c2 = y
    y, z = c2, 1.0
    for _ in range(iters):
        qs.append(z * y)
        t = (3.0 - z * y) / 2.0
        y, z = y * t, t * z
    return z * s ** -0.25, qs


def test_cn_diagonal_is_scalar_recurrence():
    lam = np.array([1e-3, 0.05, 0.4, 0.9, 1.0, 1.3])
    s, ridge, K = 1.7, 0.01, 7
    X, resid, _ = oracle.cn_inv_root(np.diag(lam)[None], np.array([s]), K, ridge=ridge)
    want = [cn_scalar(l, s, K, ridge) for l in lam]
    np.testing.assert_allclose(np.diag(X[0]), [w[0] for w in want], rtol=1e-13)
    assert np.max(np.abs(X[0] - np.diag(np.diag(X[0])))) == 0.0
    for i in range(K):
        r = math.sqrt(sum((w[1][i] - 1.0) ** 2 for w in want) / len(lam))
        assert abs(resid[0, i] - r) <= 1e-13 * max(1.0, r)


def test_cn_commuting_family():
    lam = np.linspace(0.05, 1.0, 20)
    A, Q = sym_from_spectrum(lam, 1)
    X, _, _ = oracle.cn_inv_root(A[None], np.array([1.0]), 6)
    xs = np.array([cn_scalar(l, 1.0, 6)[0] for l in lam])
    assert rel_fro(X[0], (Q * xs) @ Q.T) < 1e-12


def test_cn_converges_to_evd_and_counts():
    A = synth.wishart(3, 32, seed=8).double().numpy()
    s = np.array([np.linalg.eigvalsh(a)[-1] for a in A])
    X, resid, mm = oracle.cn_inv_root(A, s, 30)
    ref = oracle.evd_inv_root(A)
    for k in range(3):
        assert rel_fro(X[k], ref[k]) < 1e-10
    assert resid[:, -1].max() < 1e-12
    assert oracle.cn_inv_root(A[:1], s[:1], 10)[2] == 36
    assert oracle.cn_inv_root(A[:1], s[:1], 1)[2] == 0
    assert oracle.cn_inv_root(A[:1], s[:1], 2)[2] == 4


def test_cn_residual_is_residual_of_iterate():
    # resid[k] (from the M recurrence) must equal ||X_k^4 A_s - I|| computed
    # from the X recurrence alone: ties the two halves of the coupled iteration.
    A = synth.wishart(1, 24, seed=9).double().numpy()
    s = np.array([2.5])
    _, resid, _ = oracle.cn_inv_root(A, s, 6)
    As = A[0] / s[0]
    for k in range(1, 6):
        Xk = oracle.cn_inv_root(A, s, k)[0][0] * s[0] ** 0.25
        r = np.linalg.norm(np.linalg.matrix_power(Xk, 4) @ As - np.eye(24)) / math.sqrt(24)
        assert abs(r - resid[0, k]) < 1e-12


def test_ndb_diagonal_is_scalar_recurrence():
    lam = np.array([2e-3, 0.1, 0.5, 0.99, 1.0, 1.2])
    s, ridge, K = 1.3, 0.02, 6
    X, resid, _ = oracle.ndb_inv_root(np.diag(lam)[None], np.array([s]), K, ridge=ridge)
    want = [ndb_scalar(l, s, K, ridge) for l in lam]
    np.testing.assert_allclose(np.diag(X[0]), [w[0] for w in want], rtol=1e-13)
    for stage in range(2):
        for i in range(K):
            r = math.sqrt(sum((w[1][stage * K + i] - 1.0) ** 2 for w in want) / len(lam))
            assert abs(resid[0, stage, i] - r) <= 1e-13 * max(1.0, r)


def cn_scalar32(lam, s, iters, ridge):
    """Coupled Newton on one eigenvalue in numpy float32 scalars (rounding after
    every operation, as a float32 run of the matrix iteration does on a diagonal)."""
    f = np.float32
    m = (f(lam) + f(ridge)) / f(s)
    x = None
    for i in range(iters):
        t = (f(5.0) - m) / f(4.0)
        x = t if i == 0 else x * t
        if i < iters - 1:
            t2 = t * t
            m = (t2 * t2) * m
    return float(x) * s ** -0.25


def ndb_scalar32(lam, s, iters, ridge):
    """Two Newton-Schulz Denman-Beavers stages on one eigenvalue in float32 scalars."""
    f = np.float32

    def stage(c, keep_y):
        y, z = c, f(1.0)
        for i in range(iters):
            q = c if i == 0 else z * y
            t = (f(3.0) - q) / f(2.0)
            last = i == iters - 1
            yn = y * t if (not last or keep_y) else y
            zn = (t if i == 0 else t * z) if (not last or not keep_y) else z
            y, z = yn, zn
        return y if keep_y else z

    c = (f(lam) + f(ridge)) / f(s)
    return float(stage(stage(c, True), False)) * s ** -0.25


def test_float32_runs_are_float32_recurrences():
    # On a diagonal block every product of the matrix iteration is one rounded
    # scalar product, so the float32 run must reproduce the float32 scalar
    # recurrence bit for bit -- and differ from the float64 run, or it is not a
    # float32 run.
    lam = np.array([1e-5, 3e-3, 0.05, 0.4, 0.9, 1.0])
    s, ridge, K = 1.3, 1e-6, 9
    A = np.diag(lam)[None]
    x32 = oracle.cn_inv_root(A, np.array([s]), K, ridge=ridge, dtype=np.float32)[0][0]
    want = [cn_scalar32(l, s, K, ridge) for l in lam]
    np.testing.assert_array_equal(np.diag(x32), want)
    assert np.max(np.abs(x32 - np.diag(np.diag(x32)))) == 0.0
    x64 = oracle.cn_inv_root(A, np.array([s]), K, ridge=ridge)[0][0]
    assert np.any(np.diag(x32) != np.diag(x64))
    n32 = oracle.ndb_inv_root(A, np.array([s]), K, ridge=ridge, dtype=np.float32)[0][0]
    np.testing.assert_array_equal(np.diag(n32), [ndb_scalar32(l, s, K, ridge) for l in lam])
    n64 = oracle.ndb_inv_root(A, np.array([s]), K, ridge=ridge)[0][0]
    assert np.any(np.diag(n32) != np.diag(n64))
    # On a well-conditioned block the float32 run stays within float32 rounding of
    # the float64 run.
    W = synth.wishart(1, 64, seed=12).double().numpy()
    sw = np.array([np.linalg.eigvalsh(W[0])[-1]])
    for fn in (oracle.cn_inv_root, oracle.ndb_inv_root):
        assert rel_fro(fn(W, sw, 10, dtype=np.float32)[0][0], fn(W, sw, 10)[0][0]) < 1e-5


def test_ndb_commuting_family_converges_and_counts():
    lam = np.linspace(0.02, 1.0, 16)
    A, Q = sym_from_spectrum(lam, 2)
    X, _, _ = oracle.ndb_inv_root(A[None], np.array([1.0]), 5)
    xs = np.array([ndb_scalar(l, 1.0, 5)[0] for l in lam])
    assert rel_fro(X[0], (Q * xs) @ Q.T) < 1e-12
    A = synth.wishart(2, 32, seed=4).double().numpy()
    s = np.array([np.linalg.eigvalsh(a)[-1] for a in A])
    X, resid, mm = oracle.ndb_inv_root(A, s, 25)
    ref = oracle.evd_inv_root(A)
    assert max(rel_fro(X[k], ref[k]) for k in range(2)) < 1e-10
    assert mm == 2 * (3 * 25 - 3)
    assert oracle.ndb_inv_root(A[:1], s[:1], 10)[2] == 54
    assert oracle.ndb_inv_root(A[:1], s[:1], 1)[2] == 1  # stage 1 needs Y_1 = C T_0


# --------------------------------------------------------------------------- Chebyshev


@pytest.mark.parametrize("d", [1, 2, 8, 16, 32])
def test_cheb_coeffs_match_numpy_interpolation(d):
    lo, hi = 1e-2, 1.05
    c = oracle.cheb_coeffs(d, lo, hi)
    ref = npcheb.chebinterpolate(lambda t: (0.5 * (hi - lo) * t + 0.5 * (hi + lo)) ** -0.25, d)
    np.testing.assert_allclose(c, ref, rtol=1e-12, atol=1e-13)
    # Interpolates at the first-kind nodes.
    t = np.cos(np.pi * (np.arange(d + 1) + 0.5) / (d + 1))
    x = 0.5 * (hi - lo) * t + 0.5 * (hi + lo)
    np.testing.assert_allclose(npcheb.chebval(t, c), x ** -0.25, rtol=1e-12)


def test_cheb_error_decreases_with_degree():
    lo, hi = 0.05, 1.05
    x = np.linspace(lo, hi, 2001)
    t = (2 * x - lo - hi) / (hi - lo)
    errs = [np.max(np.abs(npcheb.chebval(t, oracle.cheb_coeffs(d, lo, hi)) - x ** -0.25))
            for d in (4, 8, 16, 32)]
    assert all(errs[i + 1] < errs[i] for i in range(3))
    assert errs[-1] < 1e-6


@pytest.mark.parametrize("d", [1, 2, 3, 16])
def test_cheb_matrix_matches_scalar_polynomial(d):
    lo, hi, s, ridge = 1e-2, 1.05, 1.4, 0.003
    lam = np.linspace(0.03, 1.4, 12)
    A, Q = sym_from_spectrum(lam, 3)
    X, mm = oracle.cheb_inv_root(A[None], np.array([s]), d, lo, hi, ridge=ridge)
    c = oracle.cheb_coeffs(d, lo, hi)
    t = (2 * (lam + ridge) / s - lo - hi) / (hi - lo)
    want = (Q * (s ** -0.25 * npcheb.chebval(t, c))) @ Q.T
    assert rel_fro(X[0], want) < 1e-12
    assert mm == max(d - 1, 0)
    Xd, _ = oracle.cheb_inv_root(np.diag(lam)[None], np.array([s]), d, lo, hi, ridge=ridge)
    np.testing.assert_allclose(np.diag(Xd[0]), s ** -0.25 * npcheb.chebval(t, c), rtol=1e-12)


# ------------------------------------------------------------------------ power / Frobenius


@pytest.mark.parametrize("iters", [1, 2, 3, 6])
def test_power_two_by_two_closed_form(iters):
    # A = diag(1, r), v0 = (1, 1): v after k normalised products is prop. to (1, r^k);
    # the estimate is the Rayleigh quotient of A^{iters-1} v0.
    r = 0.5
    k = iters - 1
    want = (1 + r ** (2 * k + 1)) / (1 + r ** (2 * k))
    got = oracle.power_lambda(np.diag([1.0, r])[None], np.ones((1, 2, 1)), iters)
    assert abs(got[0] - want) < 1e-15


def test_power_takes_max_over_vectors_and_ridge():
    A = np.diag([3.0, 1.0, 0.5])[None]
    V0 = np.zeros((1, 3, 2))
    V0[0, 1, 0] = 1.0  # eigenvector of 1.0: stays there
    V0[0, :, 1] = 1.0  # reaches 3.0
    got = oracle.power_lambda(A, V0, 60)
    assert abs(got[0] - 3.0) < 1e-12
    got1 = oracle.power_lambda(A, V0[:, :, :1], 5, ridge=0.25)
    assert abs(got1[0] - 1.25) < 1e-15


def test_power_brute_force_small():
    rng = np.random.default_rng(0)
    for b in (2, 5, 8):
        lam = np.sort(rng.uniform(0.1, 1.0, b))
        lam[-1] = 2.0
        A, _ = sym_from_spectrum(lam, b)
        V0 = rng.standard_normal((1, b, 4))
        got = oracle.power_lambda(A[None], V0, 80)
        assert abs(got[0] - np.linalg.eigvalsh(A)[-1]) < 1e-10
        # Never above lambda_max (a Rayleigh quotient).
        few = oracle.power_lambda(A[None], V0, 2)
        assert few[0] <= 2.0 + 1e-12


def test_frobenius():
    lam = np.array([0.1, 0.5, 2.0, 3.0])
    A, _ = sym_from_spectrum(lam, 4)
    got = oracle.frobenius_norm(A[None], ridge=0.5)
    assert abs(got[0] - math.sqrt(np.sum((lam + 0.5) ** 2))) < 1e-12
    B = np.arange(9.0).reshape(1, 3, 3)
    assert abs(oracle.frobenius_norm(B)[0] - np.linalg.norm(B[0], "fro")) < 1e-12


# ---------------------------------------------------------------------- accumulate / apply


def brute_accumulate(F, G, beta, vr, vc):
    ng, b, _ = G.shape
    out = np.zeros_like(F)
    for j in range(ng):
        for i in range(b):
            for k in range(b):
                sl = sum(G[j, i, t] * G[j, k, t] for t in range(b))
                sr = sum(G[j, t, i] * G[j, t, k] for t in range(b))
                out[j, i, k] = beta * F[j, i, k] + (1 - beta) * sl
                out[ng + j, i, k] = beta * F[ng + j, i, k] + (1 - beta) * sr
                if i >= vr[j] or k >= vr[j]:
                    out[j, i, k] = 1.0 if i == k else 0.0
                if i >= vc[j] or k >= vc[j]:
                    out[ng + j, i, k] = 1.0 if i == k else 0.0
    return out


def test_accumulate_brute_force_with_padding():
    rng = np.random.default_rng(1)
    ng, b = 3, 5
    vr, vc = [5, 3, 5], [5, 5, 2]
    G = rng.standard_normal((ng, b, b))
    for j in range(ng):
        G[j, vr[j]:, :] = 0
        G[j, :, vc[j]:] = 0
    F = rng.standard_normal((2 * ng, b, b))
    got = oracle.accumulate(F, G, 0.9, vr, vc)
    np.testing.assert_allclose(got, brute_accumulate(F, G, 0.9, vr, vc), rtol=1e-13, atol=1e-14)


def test_accumulate_two_steps_closed_form():
    rng = np.random.default_rng(2)
    G1 = rng.standard_normal((2, 4, 4))
    G2 = rng.standard_normal((2, 4, 4))
    beta = 0.95
    F = oracle.accumulate(np.zeros((4, 4, 4)), G1, beta)
    F = oracle.accumulate(F, G2, beta)
    for j in range(2):
        wl = beta * (1 - beta) * G1[j] @ G1[j].T + (1 - beta) * G2[j] @ G2[j].T
        wr = beta * (1 - beta) * G1[j].T @ G1[j] + (1 - beta) * G2[j].T @ G2[j]
        np.testing.assert_allclose(F[j], wl, rtol=1e-13)
        np.testing.assert_allclose(F[2 + j], wr, rtol=1e-13)
    # beta = 0 is the plain Gram matrices.
    F0 = oracle.accumulate(F, G1, 0.0)
    np.testing.assert_allclose(F0[1], G1[1] @ G1[1].T, rtol=1e-13)
    np.testing.assert_allclose(F0[3], G1[1].T @ G1[1], rtol=1e-13)


def test_apply_brute_force_identity_and_diagonal():
    rng = np.random.default_rng(3)
    ng, b = 2, 4
    G = rng.standard_normal((ng, b, b))
    Fr = rng.standard_normal((2 * ng, b, b))
    got = oracle.apply_preconditioner(G, Fr)
    for j in range(ng):
        for i in range(b):
            for k in range(b):
                v = sum(Fr[j, i, p] * G[j, p, q] * Fr[ng + j, q, k]
                        for p in range(b) for q in range(b))
                assert abs(got[j, i, k] - v) < 1e-12
    eye = np.broadcast_to(np.eye(b), (2 * ng, b, b))
    np.testing.assert_allclose(oracle.apply_preconditioner(G, eye), G, rtol=1e-15)
    l = np.diag([1.0, 2.0, 3.0, 4.0])
    r = np.diag([0.5, 0.25, 2.0, 1.0])
    Fd = np.stack([l, l, r, r])
    want = np.diag(l)[:, None] * G * np.diag(r)[None, :]
    np.testing.assert_allclose(oracle.apply_preconditioner(G, Fd), want, rtol=1e-14)


# ------------------------------------------------------------------------ planted mistakes


def test_planted_mistakes_are_caught():
    """Slipped versions of the scalar maps disagree with the matrix oracle."""
    lam = np.array([0.05, 0.3, 0.8])
    X, _, _ = oracle.cn_inv_root(np.diag(lam)[None], np.array([1.0]), 5)

    def cn_wrong(l, iters):  # (3I - M)/2 instead of (5I - M)/4
        m, x = l, 1.0
        for _ in range(iters):
            t = (3.0 - m) / 2.0
            x, m = x * t, m * t ** 4
        return x

    assert np.max(np.abs(np.diag(X[0]) - [cn_wrong(l, 5) for l in lam])) > 1e-3
    Xn, _, _ = oracle.ndb_inv_root(np.diag(lam)[None], np.array([1.0]), 5)
    # Keeping Y (the square root) in stage 2 gives A^{1/4}, not A^{-1/4}.
    assert np.max(np.abs(np.diag(Xn[0]) - lam ** 0.25)) > 1e-2
    # A transposed operand in apply breaks the brute-force pin for a non-symmetric G.
    rng = np.random.default_rng(5)
    G = rng.standard_normal((1, 3, 3))
    Fr = rng.standard_normal((2, 3, 3))
    U = oracle.apply_preconditioner(G, Fr)
    assert np.max(np.abs(U[0] - Fr[0] @ G[0].T @ Fr[1])) > 1e-3


def test_pack_blocks_against_numpy_block():
    """Cutting a weight into B x B blocks ([pt] Metodologia 1), pinned by numpy's own
    block assembly and hand-counted extents on a ragged 5 x 7 matrix with B = 4."""
    rng = np.random.default_rng(11)
    M = rng.standard_normal((5, 7))
    blocks, vr, vc = oracle.pack_blocks(M, 4)
    assert blocks.shape == (4, 4, 4)
    assert list(vr) == [4, 4, 1, 1] and list(vc) == [4, 3, 4, 3]  # row-block-major
    padded = np.zeros((8, 8))
    padded[:5, :7] = M
    assert np.array_equal(np.block([[blocks[0], blocks[1]], [blocks[2], blocks[3]]]), padded)
    assert np.array_equal(oracle.unpack_blocks(blocks, 5, 7), M)
    one, vr1, vc1 = oracle.pack_blocks(M[:4, :4], 4)
    assert one.shape == (1, 4, 4) and np.array_equal(one[0], M[:4, :4])
    assert list(vr1) == [4] and list(vc1) == [4]
    # A column-major enumeration (a plausible slip) puts block (1, 0) second.
    assert not np.array_equal(np.block([[blocks[0], blocks[2]], [blocks[1], blocks[3]]]), padded)


def test_update_weights_closed_forms():
    """W - lr L^{-1/4} G R^{-1/4}: identity roots give W - lr G, diagonal roots scale
    rows and columns, lr = 0 leaves W."""
    rng = np.random.default_rng(12)
    W = rng.standard_normal((2, 3, 3))
    G = rng.standard_normal((2, 3, 3))
    eye = np.broadcast_to(np.eye(3), (4, 3, 3))
    assert np.allclose(oracle.update_weights(W, G, eye, 0.1), W - 0.1 * G, rtol=0, atol=1e-15)
    assert np.array_equal(oracle.update_weights(W, G, eye, 0.0), W)
    dl = rng.uniform(0.5, 2.0, (2, 3))
    dr = rng.uniform(0.5, 2.0, (2, 3))
    Fr = np.concatenate([np.stack([np.diag(x) for x in dl]), np.stack([np.diag(x) for x in dr])])
    want = W - 0.25 * (dl[:, :, None] * G * dr[:, None, :])
    assert np.allclose(oracle.update_weights(W, G, Fr, 0.25), want, rtol=0, atol=1e-14)
