"""Float64 oracle: inverse 4th roots A^{-1/4} of stacked SPD blocks.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain NumPy in float64,
one block at a time.

The pages name four ways to get A^{-1/4} and print none of their formulas:
eigen-decomposition (the Distributed Shampoo default, [pt] Definicao do
Problema item 2), Coupled Newton ([pt] same item; [tg] "CN - Coupled Newton
Iteration"), Newton-Denman-Beavers ([pt] Metodologia 2, "Iteracao de
Newton-Denman-Beavers (NDB)") and Chebyshev polynomials evaluated with
Clenshaw's recurrence ([pt] Metodologia 2, "Aproximacoes de Polinomios de
Chebyshev").  The readings taken (each the plainest textbook form that fits
what the pages say about it):

Scaling.  Every iterative solver works on A_s = (A + ridge I) / s, where s is
the per-block scale (a power-iteration lambda_max estimate or the Frobenius
norm), so that the spectrum sits near (0, 1] ([pt] Metodologia 2: the scale
brings the eigenvalues near 1).  The result is s^{-1/4} times the solver's
root of A_s.

Coupled Newton, p = 4 (the coupled inverse p-th root iteration of Guo and
Higham, 2006).  X_0 = I, M_0 = A_s;  T_k = ((p+1) I - M_k) / p;
X_{k+1} = X_k T_k;  M_{k+1} = T_k^4 M_k, with T^4 formed as (T^2)^2.  The
iterates commute and M_k = X_k^4 A_s throughout.  Iteration 0 costs three
products (X_1 = T_0 is free) and the last iteration skips the M update (one
product), so K iterations cost 4K - 4 products.

Newton-Denman-Beavers.  The pages say NDB yields a square root and an inverse
square root together and that its first iteration is trimmed so that a step
costs three products, fewer in practice ([pt] Metodologia 2, NDB bullet).  The
matmul-only (Newton-Schulz) form of the Denman-Beavers iteration has exactly
that shape:  Y_0 = C, Z_0 = I;  T_k = (3I - Z_k Y_k) / 2;
Y_{k+1} = Y_k T_k;  Z_{k+1} = T_k Z_k;  Y -> C^{1/2}, Z -> C^{-1/2}.  At k = 0
the product Z_0 Y_0 = C and Z_1 = T_0 are free, so the first step costs one
product.  A^{-1/4} takes two such stages: stage 1 on C = A_s keeps
Y ~ A_s^{1/2}; stage 2 on C = that Y keeps Z ~ A_s^{-1/4}.  ``iters`` counts
iterations per stage; the last iteration of a stage forms only the iterate
that stage keeps, so a stage of K iterations costs 3K - 3 products.

Chebyshev / Clenshaw.  f(x) = x^{-1/4} on an interval [lo, hi] containing the
scaled spectrum is replaced by its degree-d interpolant at the d+1 Chebyshev
points of the first kind, written in the Chebyshev basis; the matrix
polynomial is evaluated by Clenshaw's recurrence on
S = (2 A_s - (lo+hi) I) / (hi - lo):  b_{d+1} = b_{d+2} = 0,
b_j = c_j I + 2 S b_{j+1} - b_{j+2} (j = d..1),  P = c_0 I + S b_1 - b_2.
b_d and b_{d-1} are combinations of I and S, so d - 1 products remain.

Residuals.  CN reports r_k = ||M_k - I||_F / sqrt(B) for k = 0..K-1 (the
residual ||X_k^4 A_s - I|| of iterate X_k); NDB reports ||Z_k Y_k - I||_F /
sqrt(B) for k = 0..K-1 of each stage.
"""

import math

import numpy as np


def _as64(x):
    return np.asarray(x, dtype=np.float64)


def _scaled(a, s, ridge, dtype=np.float64):
    b = a.shape[0]
    a = np.asarray(a, dtype=dtype)
    return (a + dtype(ridge) * np.eye(b, dtype=dtype)) / dtype(s)


def _resid(m):
    b = m.shape[0]
    return float(np.linalg.norm(m - np.eye(b), "fro") / math.sqrt(b))


def evd_inv_root(A, ridge=0.0):
    """A^{-1/4} = Q diag(lambda^{-1/4}) Q^T from a symmetric eigen-decomposition.

    The eigen-decomposition root is the default that the batched solvers
    replace ([pt] Definicao do Problema, item 2); here it is the exact answer the
    iterative solvers are measured against.
    """
    A = _as64(A)
    n, b, _ = A.shape
    out = np.empty_like(A)
    for k in range(n):
        lam, q = np.linalg.eigh(A[k] + ridge * np.eye(b))
        if np.min(lam) <= 0.0:
            raise ValueError("block %d is not positive definite" % k)
        out[k] = (q * lam ** -0.25) @ q.T
    return out


def cn_inv_root(A, scale, iters, ridge=0.0, dtype=np.float64):
    """Coupled Newton inverse 4th root of every block (reading in module docstring).

    Returns (X, resid, matmuls): X (N, B, B) ~ A^{-1/4}; resid (N, iters) with
    resid[k, i] = ||M_i - I||_F / sqrt(B); matmuls = products per block.
    dtype np.float32 runs the same steps in plain round-to-nearest float32 (the
    scaled block, every product and every iterate), which shows what ordinary
    arithmetic of that precision can deliver on a given block.
    """
    A = _as64(A)
    scale = _as64(scale)
    n, b, _ = A.shape
    p = 4.0
    eye = np.eye(b, dtype=dtype)
    X_out = np.empty_like(A)
    resid = np.empty((n, iters))
    mm = 0
    for k in range(n):
        M = _scaled(A[k], scale[k], ridge, dtype)
        X = eye.copy()
        mm = 0
        for i in range(iters):
            resid[k, i] = _resid(M)
            T = ((p + 1.0) * eye - M) / p
            if i == 0:
                X = T
            else:
                X = X @ T
                mm += 1
            if i < iters - 1:
                T2 = T @ T
                T4 = T2 @ T2
                M = T4 @ M
                mm += 3
        X_out[k] = scale[k] ** -0.25 * X
    return X_out, resid, mm


def _ndb_stage(C, iters, keep):
    """One Newton-Schulz Denman-Beavers stage on C; keep is "Y" or "Z".

    Runs in C's dtype.  Returns (kept iterate, residual list, products used)."""
    b = C.shape[0]
    eye = np.eye(b, dtype=C.dtype)
    Y = C
    Z = eye
    res = []
    mm = 0
    for i in range(iters):
        last = i == iters - 1
        if i == 0:
            P = C
        else:
            P = Z @ Y
            mm += 1
        res.append(_resid(P))
        T = (3.0 * eye - P) / 2.0
        want_y = (not last) or keep == "Y"
        want_z = (not last) or keep == "Z"
        Y_new, Z_new = Y, Z
        if want_y:
            Y_new = Y @ T
            mm += 1
        if want_z:
            if i == 0:
                Z_new = T
            else:
                Z_new = T @ Z
                mm += 1
        Y, Z = Y_new, Z_new
    return (Y if keep == "Y" else Z), res, mm


def ndb_inv_root(A, scale, iters, ridge=0.0, dtype=np.float64):
    """Two-stage Newton-Denman-Beavers inverse 4th root (reading in module docstring).

    Returns (X, resid, matmuls): resid (N, 2, iters); matmuls per block for both
    stages together.  dtype as for cn_inv_root.
    """
    A = _as64(A)
    scale = _as64(scale)
    n, b, _ = A.shape
    X_out = np.empty_like(A)
    resid = np.empty((n, 2, iters))
    mm = 0
    for k in range(n):
        As = _scaled(A[k], scale[k], ridge, dtype)
        Yh, r1, m1 = _ndb_stage(As, iters, "Y")  # ~ A_s^{1/2}
        Zq, r2, m2 = _ndb_stage(Yh, iters, "Z")  # ~ (A_s^{1/2})^{-1/2}
        resid[k, 0] = r1
        resid[k, 1] = r2
        mm = m1 + m2
        X_out[k] = scale[k] ** -0.25 * Zq
    return X_out, resid, mm


def cheb_coeffs(degree, lo, hi):
    """Chebyshev-basis coefficients c_0..c_d of the degree-d interpolant of
    x^{-1/4} at the first-kind Chebyshev points of [lo, hi] (c_0 already halved)."""
    d = int(degree)
    npts = d + 1
    t = np.array([math.cos(math.pi * (i + 0.5) / npts) for i in range(npts)])
    x = 0.5 * (hi - lo) * t + 0.5 * (hi + lo)
    fx = x ** -0.25
    c = np.empty(npts)
    for j in range(npts):
        c[j] = (2.0 / npts) * sum(
            fx[i] * math.cos(j * math.pi * (i + 0.5) / npts) for i in range(npts)
        )
    c[0] *= 0.5
    return c


def cheb_inv_root(A, scale, degree, lo, hi, ridge=0.0):
    """Chebyshev-Clenshaw inverse 4th root (reading in module docstring).

    Returns (X, matmuls)."""
    A = _as64(A)
    scale = _as64(scale)
    n, b, _ = A.shape
    d = int(degree)
    assert d >= 1
    c = cheb_coeffs(d, lo, hi)
    eye = np.eye(b)
    X_out = np.empty_like(A)
    mm = 0
    for k in range(n):
        As = _scaled(A[k], scale[k], ridge)
        S = (2.0 * As - (lo + hi) * eye) / (hi - lo)
        mm = 0
        # b_next1 = b_{j+1}, b_next2 = b_{j+2}; track whether b_{j+1} is a
        # multiple of I (then S b_{j+1} needs no product).
        b1 = np.zeros((b, b))
        b2 = np.zeros((b, b))
        b1_is_scalar = True
        b1_scalar = 0.0
        for j in range(d, 0, -1):
            if b1_is_scalar:
                Sb = b1_scalar * S
            else:
                Sb = S @ b1
                mm += 1
            bj = c[j] * eye + 2.0 * Sb - b2
            b2 = b1
            b1 = bj
            b1_is_scalar = j == d
            b1_scalar = c[j]
        if b1_is_scalar:
            Sb = b1_scalar * S
        else:
            Sb = S @ b1
            mm += 1
        P = c[0] * eye + Sb - b2
        X_out[k] = scale[k] ** -0.25 * P
    return X_out, mm
