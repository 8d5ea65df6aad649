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
