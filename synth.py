"""Seeded synthetic inputs shaped like the DASH workloads.

This module only draws inputs.  It holds none of the preconditioner's
arithmetic, so both the float64 oracle (through the tests) and the GPU library
(through the tests and ``bench.py``) may be fed from it.

Recipes (all seeded; torch's generator on the requested device, so a seed
gives different numbers on CPU and GPU -- parity tests therefore always hand the
oracle the exact fp32 bits the GPU consumed):

* ``wishart``: A_k = G_k G_k^T / c + ridge I with G_k (B x c) i.i.d. N(0, 1),
  symmetrised exactly as (A + A^T) / 2.  With c = 2B the spectrum of G G^T / c
  follows Marchenko-Pastur with ratio 1/2, roughly [0.086, 2.91].
* ``prescribed_spectrum``: A_k = Q_k diag(lam) Q_k^T, Q_k from the QR
  factorisation of a Gaussian matrix with the signs of R's diagonal folded into
  Q; lam log-uniform on [lo, hi] with both end points present; one spectrum is
  shared by all blocks.
* ``llama_layer_blocks``: gradient blocks of Llama-style transformer layers
  (d = 2048): four 2048 x 2048 attention weights and three 2048 x 5632 MLP
  weights per layer, cut into bs x bs blocks (bs = 1024), the last 512-wide
  column block of each MLP weight zero-padded; entries i.i.d. N(0, var).
  Blocks are ordered layer, weight, row block, column block.
* ``start_vectors``: power-iteration start vectors, i.i.d. N(0, 1).
* ``two_cluster_blocks``: A_k = Q_k diag(lam_k) Q_k^T (Q_k as in
  ``prescribed_spectrum``); even k: lam uniform on [0.5, 1] (kappa 2); odd k: half
  of lam at 1, half at 1e-4 (kappa 1e4, with a gap that the shifted power
  iteration resolves quickly).  Consecutive blocks thus fall into different
  solver tiers.
"""

import torch

LLAMA_D = 2048
LLAMA_FF = 5632


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def wishart(n, b, seed, cols=None, ridge=1e-6, device="cpu", chunk=64):
    """(n, b, b) fp32 stack of G G^T / cols + ridge I, G (b x cols) ~ N(0, 1)."""
    cols = 2 * b if cols is None else cols
    g = _gen(seed, device)
    out = torch.empty((n, b, b), dtype=torch.float32, device=device)
    eye = torch.eye(b, dtype=torch.float32, device=device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        G = torch.randn((e - s, b, cols), generator=g, dtype=torch.float32, device=device)
        A = torch.bmm(G, G.transpose(1, 2)) / cols + ridge * eye
        out[s:e] = 0.5 * (A + A.transpose(1, 2))
    return out


def log_uniform_spectrum(b, seed, lo=1e-6, hi=1.0):
    """b eigenvalues 10^U(log10 lo, log10 hi), sorted, end points set to lo and hi."""
    g = _gen(seed, "cpu")
    u = torch.rand((b,), generator=g, dtype=torch.float64)
    lam = torch.pow(10.0, torch.log10(torch.tensor(lo, dtype=torch.float64))
                    + u * (torch.log10(torch.tensor(hi, dtype=torch.float64))
                           - torch.log10(torch.tensor(lo, dtype=torch.float64))))
    lam, _ = torch.sort(lam)
    lam[0] = lo
    lam[-1] = hi
    return lam


def prescribed_spectrum(n, b, seed, lo=1e-6, hi=1.0, device="cpu"):
    """Returns (A (n,b,b) fp32, Q (n,b,b) fp64 on cpu, lam (b,) fp64 on cpu)."""
    lam = log_uniform_spectrum(b, seed + 7, lo, hi)
    g = _gen(seed, "cpu")
    Z = torch.randn((n, b, b), generator=g, dtype=torch.float64)
    Q, R = torch.linalg.qr(Z)
    sgn = torch.sign(torch.diagonal(R, dim1=1, dim2=2))
    sgn[sgn == 0] = 1.0
    Q = Q * sgn[:, None, :]
    A = (Q * lam[None, None, :]) @ Q.transpose(1, 2)
    A = 0.5 * (A + A.transpose(1, 2))
    return A.to(torch.float32).to(device), Q, lam


def two_cluster_blocks(n, b, seed, device="cpu"):
    """(n, b, b) fp32 blocks alternating between kappa 2 and kappa 1e4 (see above);
    drawn and formed in float64 on `device`."""
    g = _gen(seed, device)
    out = torch.empty((n, b, b), dtype=torch.float32, device=device)
    for k in range(n):
        Z = torch.randn((b, b), generator=g, dtype=torch.float64, device=device)
        Q, R = torch.linalg.qr(Z)
        sgn = torch.sign(torch.diagonal(R))
        sgn[sgn == 0] = 1.0
        Q = Q * sgn[None, :]
        if k % 2 == 0:
            lam = 0.5 + 0.5 * torch.rand(b, generator=g, dtype=torch.float64, device=device)
        else:
            lam = torch.cat([torch.ones(b // 2, dtype=torch.float64, device=device),
                             torch.full((b - b // 2,), 1e-4, dtype=torch.float64,
                                        device=device)])
        A = (Q * lam[None, :]) @ Q.T
        out[k] = (0.5 * (A + A.T)).to(torch.float32)
    return out


def llama_weight_shapes(layers=1):
    """(rows, cols) of every preconditioned weight, in block order."""
    shapes = []
    for _ in range(layers):
        shapes += [(LLAMA_D, LLAMA_D)] * 4
        shapes += [(LLAMA_D, LLAMA_FF)] * 3
    return shapes


def llama_block_layout(layers=1, bs=1024):
    """Per-block (valid_rows, valid_cols) for the Llama-layer cut; length Ng."""
    vr, vc = [], []
    for rows, cols in llama_weight_shapes(layers):
        for r0 in range(0, rows, bs):
            for c0 in range(0, cols, bs):
                vr.append(min(bs, rows - r0))
                vc.append(min(bs, cols - c0))
    return vr, vc


def llama_layer_blocks(layers, seed, var=1e-2, bs=1024, dtype=torch.bfloat16,
                       device="cpu"):
    """(Ng, bs, bs) gradient blocks plus int32 valid_rows / valid_cols tensors."""
    vr, vc = llama_block_layout(layers, bs)
    ng = len(vr)
    g = _gen(seed, device)
    G = torch.empty((ng, bs, bs), dtype=dtype, device=device)
    std = float(var) ** 0.5
    chunk = 64
    for s in range(0, ng, chunk):
        e = min(ng, s + chunk)
        G[s:e] = (std * torch.randn((e - s, bs, bs), generator=g, dtype=torch.float32,
                                    device=device)).to(dtype)
    for j in range(ng):
        if vr[j] < bs:
            G[j, vr[j]:, :] = 0
        if vc[j] < bs:
            G[j, :, vc[j]:] = 0
    return (G, torch.tensor(vr, dtype=torch.int32, device=device),
            torch.tensor(vc, dtype=torch.int32, device=device))


def start_vectors(n, b, nv, seed, device="cpu"):
    """(n, b, nv) fp32 power-iteration start vectors ~ N(0, 1)."""
    g = _gen(seed, device)
    return torch.randn((n, b, nv), generator=g, dtype=torch.float32, device=device)
