"""Pins for the solver-selection oracle (oracle/select64.py), on the CPU.

Each check rests on something other than the oracle itself: a closed form worked
out by hand for a 2 x 2 diagonal block, the Rayleigh-quotient bound, a spectrum
built with a known gap, the tier rule's boundaries, and LAPACK's eigenvalues and
eigen-decomposition root."""

import numpy as np
import pytest

import oracle
import synth


def test_lambda_min_closed_form_diagonal():
    """A = diag(a, b), v0 = (1, 1), shift c: the shifted block is diag(d1, d2) with
    d_i = c - (a_i + ridge).  After n products the Rayleigh quotient of the last
    vector is (d1^(2n-1) + d2^(2n-1)) / (d1^(2n-2) + d2^(2n-2))."""
    a, b, ridge, c = 1.0, 0.25, 0.05, 1.2
    A = np.diag([a, b])[None]
    V0 = np.ones((1, 2, 1))
    d1, d2 = c - (a + ridge), c - (b + ridge)
    for n in (1, 2, 3, 7):
        mu = (d1 ** (2 * n - 1) + d2 ** (2 * n - 1)) / (d1 ** (2 * n - 2) + d2 ** (2 * n - 2))
        got = oracle.lambda_min_estimate(A, np.array([c]), V0, n, ridge=ridge)[0]
        assert got == pytest.approx(c - mu, rel=0, abs=1e-15), n


@pytest.mark.parametrize("iters", [1, 3, 10])
def test_lambda_min_is_an_upper_bound(iters):
    """A Rayleigh quotient of c I - A' never exceeds c - lambda_min(A'), so the
    estimate is never below the true smallest eigenvalue, at any iteration count."""
    A = synth.wishart(4, 96, seed=31).double().numpy()
    V0 = synth.start_vectors(4, 96, 8, seed=32).double().numpy()
    ridge = 1e-3
    lam = oracle.power_lambda(A, V0, 10, ridge=ridge)
    est = oracle.lambda_min_estimate(A, lam, V0, iters, ridge=ridge)
    true_min = np.linalg.eigvalsh(A + ridge * np.eye(96)).min(axis=1)
    assert np.all(est >= true_min - 1e-12 * lam)


def test_lambda_min_converges_on_a_gapped_spectrum():
    """Q diag(lambda) Q^T with lambda_min = 1e-3 and every other eigenvalue in
    [0.5, 1]: the shifted iteration's ratio is about 1/2 per product, so 40
    products resolve lambda_min to far better than 1e-6 relative."""
    rng = np.random.default_rng(33)
    b = 64
    q, _ = np.linalg.qr(rng.standard_normal((b, b)))
    lam = np.concatenate([[1e-3], np.linspace(0.5, 1.0, b - 1)])
    A = ((q * lam) @ q.T)[None]
    A = 0.5 * (A + A.transpose(0, 2, 1))
    V0 = rng.standard_normal((1, b, 4))
    lmax = oracle.power_lambda(A, V0, 40)
    est = oracle.lambda_min_estimate(A, lmax, V0, 40)[0]
    assert abs(est - 1e-3) / 1e-3 < 1e-6


def test_condition_estimate_and_tier_boundaries():
    assert np.array_equal(oracle.condition_estimate([2.0, 2.0, 2.0], [0.5, 0.0, -1.0]),
                          [4.0, np.inf, np.inf])
    # A non-positive (or NaN) lambda_max is no estimate of an SPD block: inf, not a
    # small or negative kappa that would pick the cheapest tier.
    assert np.array_equal(oracle.condition_estimate([-2.0, 0.0, np.nan], [0.5, 0.5, 0.5]),
                          [np.inf, np.inf, np.inf])
    t0 = oracle.DEFAULT_TIERS[0]
    edge = 4.0 * t0["gate"] / t0["u"]          # kappa u / 4 == gate: admissible
    got = oracle.select_tiers([1.0, edge, np.nextafter(edge, np.inf), 1e12, np.inf, np.nan])
    assert got.tolist() == [0, 0, 1, 1, 1, 1]
    tiers = (
        {"solver": "cn", "prec": "fp16", "iters": 10, "u": 2.0 ** -11, "gate": 1e-2},
        {"solver": "cn", "prec": "tf32", "iters": 16, "u": 2.0 ** -11, "gate": 2e-3},
        {"solver": "ndb", "prec": "3xtf32", "iters": 12, "u": 2.0 ** -24, "gate": 1e-4},
    )
    # The middle tier has a tighter gate than the first, so it is never admissible
    # where the first is not: the rule falls through to the last tier.
    assert oracle.select_tiers([50.0, 100.0, 1e9], tiers).tolist() == [0, 2, 2]


def test_auto_root_picks_and_solves_per_block():
    """A well-conditioned Wishart block (kappa about 34) and a block with kappa
    1e6: the pipeline picks the FP16 tier for the first and the fp32-class tier for
    the second, and each root matches the eigen-decomposition root."""
    b = 64
    rng = np.random.default_rng(34)
    W = synth.wishart(1, b, seed=35).double().numpy()[0]
    q, _ = np.linalg.qr(rng.standard_normal((b, b)))
    ill = (q * np.logspace(-6, 0, b)) @ q.T
    A = np.stack([W, 0.5 * (ill + ill.T)])
    V0 = synth.start_vectors(2, b, 32, seed=36).double().numpy()
    lam = oracle.power_lambda(A, V0, 10)
    lmin = oracle.lambda_min_estimate(A, lam, V0, 40)
    kappa = oracle.condition_estimate(lam, lmin)
    choice = oracle.select_tiers(kappa)
    assert choice.tolist() == [0, 1], kappa
    X = oracle.auto_inv_root(A, lam, choice)
    ex = oracle.evd_inv_root(A)
    err = np.linalg.norm(X - ex, axis=(1, 2)) / np.linalg.norm(ex, axis=(1, 2))
    assert err[0] < 1e-8 and err[1] < 1e-8, err
    # Each block is exactly its tier's solver with that tier's iteration count.
    assert np.array_equal(X[1], oracle.cn_inv_root(A[1:], lam[1:], 24)[0][0])
    assert np.array_equal(X[0], oracle.cn_inv_root(A[:1], lam[:1], 10)[0][0])


def test_planted_mistakes_fail_the_pins():
    """Slipped versions of the selection steps disagree with what the pins fix."""
    a, b, ridge, c = 1.0, 0.25, 0.05, 1.2
    A = np.diag([a, b])[None]
    V0 = np.ones((1, 2, 1))
    got = oracle.lambda_min_estimate(A, np.array([c]), V0, 3, ridge=ridge)[0]
    # Dropping the ridge from the shift, or returning mu instead of c - mu.
    no_ridge = oracle.lambda_min_estimate(A, np.array([c]), V0, 3, ridge=0.0)[0]
    assert abs(no_ridge - got) > 1e-3
    mu = c - got
    assert abs(mu - got) > 1e-3
    # kappa u / 2 instead of kappa u / 4 moves the tier boundary.
    t0 = oracle.DEFAULT_TIERS[0]
    edge = 4.0 * t0["gate"] / t0["u"]
    assert edge * t0["u"] / 2.0 > t0["gate"] and oracle.select_tiers([edge])[0] == 0
