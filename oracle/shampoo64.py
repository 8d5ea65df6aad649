"""Float64 oracle: factor accumulation, spectral scaling and the preconditioned update.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain NumPy in float64,
one block at a time, no blocking or fusion.

Readings of the pages taken here (the pages give no formulas):

* Accumulation.  Shampoo keeps two factors built from gradient products,
  L from G G^T and R from G^T G, and raises both to the -1/4 power
  ([tg], second paragraph).  The factors are exponential moving averages with
  coefficient beta:  L <- beta L + (1-beta) G G^T,  R <- beta R + (1-beta) G^T G.
  A block whose gradient is zero-padded beyond ``valid_rows`` rows (for L) or
  ``valid_cols`` columns (for R) has its padded rows and columns reset to the
  identity after every update: zero off the diagonal, one on it.

* Stacking.  Independent B x B blocks are stacked into one (N, B, B) array and
  processed together ([pt] Metodologia 1, "Empilhamento de Tensores 3D");
  the L and R factors of all blocks share one stack, L first ([tg], the
  paragraph on block-diagonal preconditioners).  Block j of the gradient stack
  owns factor j (its L) and factor Ng + j (its R).

* Spectral scaling.  lambda_max is estimated by power iteration run from up to
  32 start vectors at once and read off as a Rayleigh quotient ([pt]
  Metodologia 2, "Multi-Power-Iteration para Escalonamento"; [tg], the
  paragraph on Frobenius vs spectral scaling).  Reading: the start vectors are
  independent columns (no orthogonalisation); each of ``iters`` steps forms
  W = A V; the columns of W are normalised to unit 2-norm except on the last
  step, where the estimate is max_j (v_j . w_j) / (v_j . v_j).  ``iters``
  therefore counts products with A.

* Preconditioned update.  U = L^{-1/4} G R^{-1/4}, the standard Shampoo
  update that the -1/4 roots of L and R exist for ([tg], second paragraph).

* Blocks of a weight.  A weight-shaped gradient (rows x cols) is cut into B x B
  blocks G_ij ([pt] Metodologia 1, "Empilhamento de Tensores 3D"), enumerated
  row-block-major (i outer, j inner); the last block row / column of a dimension
  that is not a multiple of B is zero-padded and its valid extent recorded.

* Weight step.  The pages give no optimizer update rule; the plain reading is the
  step along the preconditioned direction, W <- W - lr U, block by block.
"""

import numpy as np


def _as64(x):
    return np.asarray(x, dtype=np.float64)


def accumulate(F, G, beta, valid_rows=None, valid_cols=None):
    """One EMA update of the stacked factors; returns the new (2Ng, B, B) stack.

    F: (2Ng, B, B) factors, L_0..L_{Ng-1} then R_0..R_{Ng-1}.
    G: (Ng, B, B) gradient blocks.
    valid_rows / valid_cols: per-block counts of non-padded rows / columns of G
    (None means all B are valid).  Restates the EMA reading in the module
    docstring ([tg] second paragraph; [pt] Metodologia 1).
    """
    F = _as64(F)
    G = _as64(G)
    ng, b, _ = G.shape
    assert F.shape == (2 * ng, b, b)
    out = np.empty_like(F)
    for j in range(ng):
        g = G[j]
        out[j] = beta * F[j] + (1.0 - beta) * (g @ g.T)
        out[ng + j] = beta * F[ng + j] + (1.0 - beta) * (g.T @ g)
        vr = b if valid_rows is None else int(valid_rows[j])
        vc = b if valid_cols is None else int(valid_cols[j])
        _reset_padding(out[j], vr)
        _reset_padding(out[ng + j], vc)
    return out


def _reset_padding(f, valid):
    """Rows and columns >= valid become those of the identity."""
    b = f.shape[0]
    if valid >= b:
        return
    f[valid:, :] = 0.0
    f[:, valid:] = 0.0
    for i in range(valid, b):
        f[i, i] = 1.0


def frobenius_norm(A, ridge=0.0):
    """||A_k + ridge I||_F for every block: the Frobenius scaling the pages
    contrast with power-iteration scaling ([pt] Definicao do Problema, item 3)."""
    A = _as64(A)
    n, b, _ = A.shape
    out = np.empty(n)
    for k in range(n):
        a = A[k] + ridge * np.eye(b)
        out[k] = np.sqrt(np.sum(a * a))
    return out


def power_lambda(A, V0, iters, ridge=0.0):
    """Multi-vector power-iteration estimate of lambda_max for every block.

    A: (N, B, B) symmetric blocks; V0: (N, B, nv) start vectors (nv <= 32);
    iters >= 1 products with A.  Returns (N,) estimates.
    [pt] Metodologia 2, "Multi-Power-Iteration"; [tg] Rayleigh-quotient paragraph.
    """
    A = _as64(A)
    V0 = _as64(V0)
    n, b, _ = A.shape
    assert iters >= 1
    out = np.empty(n)
    for k in range(n):
        a = A[k] + ridge * np.eye(b)
        v = V0[k].copy()
        for it in range(iters):
            w = a @ v
            if it == iters - 1:
                num = np.sum(v * w, axis=0)
                den = np.sum(v * v, axis=0)
                out[k] = np.max(num / den)
            else:
                v = w / np.sqrt(np.sum(w * w, axis=0))
    return out


def apply_preconditioner(G, Froot):
    """U_j = Lroot_j G_j Rroot_j with Lroot_j = Froot[j], Rroot_j = Froot[Ng+j].
    [tg] second paragraph (the -1/4 powers of L and R precondition G)."""
    G = _as64(G)
    Froot = _as64(Froot)
    ng = G.shape[0]
    out = np.empty_like(G)
    for j in range(ng):
        out[j] = Froot[j] @ G[j] @ Froot[ng + j]
    return out


def pack_blocks(M, b):
    """Cut a (rows, cols) matrix into row-block-major (b, b) blocks, zero-padded.

    Returns (blocks (nbr * nbc, b, b), valid_rows (nbr * nbc,), valid_cols
    (nbr * nbc,)) with nbr = ceil(rows / b), nbc = ceil(cols / b); block i * nbc + j
    holds rows i*b.. and columns j*b.. of M ([pt] Metodologia 1).
    """
    M = _as64(M)
    rows, cols = M.shape
    nbr = -(-rows // b)
    nbc = -(-cols // b)
    blocks = np.zeros((nbr * nbc, b, b))
    vr = np.zeros(nbr * nbc, dtype=np.int64)
    vc = np.zeros(nbr * nbc, dtype=np.int64)
    for i in range(nbr):
        for j in range(nbc):
            k = i * nbc + j
            r = min(b, rows - i * b)
            c = min(b, cols - j * b)
            blocks[k, :r, :c] = M[i * b:i * b + r, j * b:j * b + c]
            vr[k] = r
            vc[k] = c
    return blocks, vr, vc


def unpack_blocks(blocks, rows, cols):
    """Inverse of pack_blocks: the (rows, cols) matrix, padding dropped."""
    blocks = _as64(blocks)
    b = blocks.shape[1]
    nbc = -(-cols // b)
    M = np.empty((rows, cols))
    for k in range(blocks.shape[0]):
        i, j = divmod(k, nbc)
        r = min(b, rows - i * b)
        c = min(b, cols - j * b)
        M[i * b:i * b + r, j * b:j * b + c] = blocks[k, :r, :c]
    return M


def update_weights(W, G, Froot, lr):
    """W_j - lr U_j for every block, U from apply_preconditioner (the weight-step
    reading in the module docstring)."""
    return _as64(W) - lr * apply_preconditioner(G, Froot)
