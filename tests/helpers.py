"""Test-side helpers: library fixture, TF32 rounding on the host, error norms."""

import numpy as np
import pytest
import torch


def rel_fro(x, y):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    return float(np.linalg.norm(x - y) / np.linalg.norm(y))


def rel_fro_blocks(x, y):
    """Relative Frobenius error of each block of two (N, B, B) stacks."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    return np.linalg.norm((x - y).reshape(len(x), -1), axis=1) / np.linalg.norm(
        y.reshape(len(y), -1), axis=1)


def rna_tf32(t):
    """Round fp32 values to TF32 (10 explicit mantissa bits), ties away from zero."""
    bits = t.contiguous().view(torch.int32)
    bits = (bits + 0x1000) & ~0x1FFF
    return bits.view(torch.float32)


def split_tf32(t):
    hi = rna_tf32(t)
    lo = rna_tf32(t - hi)
    return hi, lo


def to64(t):
    return t.detach().double().cpu().numpy()


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def library():
    """Build (if stale) and load libdashroot.so; fails loudly when it cannot."""
    from matrix_inverse_roots_gb300 import build as b
    import matrix_inverse_roots_gb300 as dr

    b.build()
    dr.load_library()
    return dr


STORE_DTYPES = {"3xtf32": torch.float32, "tf32": torch.float32, "fp16": torch.float16,
                "bf16": torch.bfloat16}


def _rd(x, dt):
    return x.to(dt).float()


def cn_emulated(a, s, iters, prec, ridge=0.0):
    """Coupled Newton on the CPU with the library's storage rule: every iterate is
    rounded to the precision's storage type, products and epilogue algebra run in
    float32.  Used only to show what arithmetic of that precision can deliver."""
    dt = STORE_DTYPES[prec]
    a = a.float()
    b = a.shape[0]
    eye = torch.eye(b, dtype=torch.float32)
    As = (a + ridge * eye) / s
    M = _rd(As, dt)
    T = _rd((5 * eye - As) / 4, dt)
    X = T
    for i in range(iters):
        if i > 0:
            X = _rd(X @ T, dt)
        if i < iters - 1:
            T2 = _rd(T @ T, dt)
            T4 = _rd(T2 @ T2, dt)
            C = T4 @ M
            M = _rd(C, dt)
            T = _rd((5 * eye - C) / 4, dt)
    if iters == 1:
        X = _rd((5 * eye - As) / 4, dt)
    return (X * s ** -0.25).double().numpy()


def ndb_emulated(a, s, iters, prec, ridge=0.0):
    """Two-stage Newton-Denman-Beavers on the CPU with the library's storage rule."""
    dt = STORE_DTYPES[prec]
    a = a.float()
    b = a.shape[0]
    eye = torch.eye(b, dtype=torch.float32)

    def stage(Cexact, keep_y):
        C = _rd(Cexact, dt)
        Y, Z = C, _rd((3 * eye - Cexact) / 2, dt)
        T = Z
        for i in range(iters):
            if i > 0:
                P = Z @ Y
                T = _rd((3 * eye - P) / 2, dt)
            last = i == iters - 1
            Yn = _rd(Y @ T, dt) if (not last or keep_y) else Y
            Zn = (T if i == 0 else _rd(T @ Z, dt)) if (not last or not keep_y) else Z
            Y, Z = Yn, Zn
        return Y if keep_y else Z

    return (stage(stage((a + ridge * eye) / s, True), False) * s ** -0.25).double().numpy()
