"""Per-block solver selection by a condition estimate: float64 oracle.

Test infrastructure, like the rest of this package: only the tests, the smoke
check and the benchmark's CPU baseline may import it.

Source: [pt] Significancia e Alegacoes, item Direcoes Futuras: choosing the
solver per block from the block's condition number is named there as a direction
for future work.  The pages give no rule, so everything below is a reading (each
step says which):

1. Condition estimate.  lambda_max comes from the multi-vector power iteration
   (shampoo64.power_lambda).  lambda_min is estimated by the same iteration on the
   shifted block c I - (A + ridge I) with c = the lambda_max estimate: its largest
   eigenvalue is c - lambda_min, so lambda_min_hat = c - mu_hat.  A Rayleigh
   quotient never exceeds the largest eigenvalue, so mu_hat <= c - lambda_min and
   lambda_min_hat >= lambda_min for every iteration count: the estimate errs
   towards a better-conditioned block, and kappa_hat = lambda_max_hat /
   lambda_min_hat <= kappa.  A non-positive lambda_min_hat (no resolved gap) or
   lambda_max_hat (no usable estimate of an SPD block) gives kappa_hat = inf.
2. Tiers.  An ordered list, cheapest first, of (solver, precision, iterations,
   unit roundoff u, error gate).  Storing the scaled block at roundoff u moves its
   smallest eigenvalue, about 1/kappa, by about kappa u relative, and its inverse
   4th root by a quarter of that; a tier is admissible when kappa_hat u / 4 <= its
   gate.  The first admissible tier is chosen, the last (most accurate) tier when
   none is.
3. The root of each block is that tier's solver with that tier's iteration count,
   scaled by lambda_max_hat as in the fixed-solver path.  In float64 the tier's
   precision does not change the arithmetic: it only sets the gate a GPU result of
   that block is held to.
"""

import math

import numpy as np

from .roots64 import cheb_inv_root, cn_inv_root, ndb_inv_root
from .shampoo64 import power_lambda

U_FP16 = 2.0 ** -11
U_FP32 = 2.0 ** -24

# Cheapest first.  CN is the cheaper solver per iteration (4 products against 6);
# 24 iterations take Coupled Newton from a smallest scaled eigenvalue of 1e-6 to
# convergence (each early iteration multiplies it by about (5/4)^4).
DEFAULT_TIERS = (
    {"solver": "cn", "prec": "fp16", "iters": 10, "u": U_FP16, "gate": 1e-2},
    {"solver": "cn", "prec": "3xtf32", "iters": 24, "u": U_FP32, "gate": 1e-4},
)


def _as64(x):
    return np.asarray(x, dtype=np.float64)


def lambda_min_estimate(A, lam_max, V0, iters, ridge=0.0):
    """lambda_min_hat per block: power iteration on c I - (A + ridge I), c = lam_max.

    A (N, B, B) symmetric; lam_max (N,) the lambda_max estimates; V0 (N, B, nv) the
    start vectors; iters >= 1 products.  Returns (N,) estimates (reading 1)."""
    A = _as64(A)
    lam_max = _as64(lam_max)
    n, b, _ = A.shape
    eye = np.eye(b)
    shifted = np.stack([lam_max[k] * eye - (A[k] + ridge * eye) for k in range(n)])
    mu = power_lambda(shifted, V0, iters)
    return lam_max - mu


def condition_estimate(lam_max, lam_min):
    """kappa_hat = lam_max / lam_min per block, inf unless both are positive
    (reading 1)."""
    lam_max = _as64(lam_max)
    lam_min = _as64(lam_min)
    out = np.full(lam_max.shape, np.inf)
    ok = (lam_min > 0) & (lam_max > 0)
    out[ok] = lam_max[ok] / lam_min[ok]
    return out


def select_tiers(kappa, tiers=DEFAULT_TIERS):
    """Index of the chosen tier for every block (reading 2)."""
    kappa = _as64(kappa)
    out = np.empty(kappa.shape, dtype=np.int64)
    for i, k in enumerate(kappa.ravel()):
        choice = len(tiers) - 1
        if not math.isnan(k):
            for t, tier in enumerate(tiers):
                if k * tier["u"] / 4.0 <= tier["gate"]:
                    choice = t
                    break
        out.flat[i] = choice
    return out


def auto_inv_root(A, lam_max, choice, tiers=DEFAULT_TIERS, ridge=0.0, cheb=(1e-2, 1.05)):
    """A^{-1/4} of every block by its chosen tier's solver (reading 3).

    choice (N,) tier indices from select_tiers; cheb (lo, hi) is the interval of a
    Chebyshev tier, whose "iters" is its degree.  Returns (N, B, B)."""
    A = _as64(A)
    lam_max = _as64(lam_max)
    n = A.shape[0]
    X = np.empty_like(A)
    for k in range(n):
        tier = tiers[int(choice[k])]
        a, s = A[k:k + 1], lam_max[k:k + 1]
        if tier["solver"] == "cn":
            X[k] = cn_inv_root(a, s, tier["iters"], ridge=ridge)[0][0]
        elif tier["solver"] == "ndb":
            X[k] = ndb_inv_root(a, s, tier["iters"], ridge=ridge)[0][0]
        elif tier["solver"] == "cheb":
            X[k] = cheb_inv_root(a, s, tier["iters"], cheb[0], cheb[1], ridge=ridge)[0][0]
        else:
            raise ValueError(tier["solver"])
    return X
