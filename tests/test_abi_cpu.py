"""Host-side checks of the C ABI: the library builds, loads and exports every
declared entry point, and rejects bad arguments before touching a GPU."""

import ctypes
import os
import re

import pytest

import oracle
from tests.helpers import library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "dashroot.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    dr = library()
    lib = dr.load_library()
    names = declared_functions()
    assert len(names) >= 12, names
    for n in names:
        assert hasattr(lib, n), "missing export %s" % n
    assert set(names) == set(dr.SYMBOLS)
    assert "sm_103a" in dr.version()


def test_status_strings():
    dr = library()
    for s in range(7):
        assert dr.status_string(s).startswith("DASH_")


def test_matmul_counts_match_oracle():
    dr = library()
    import numpy as np

    A = np.eye(4)[None] * 0.5
    s = np.array([1.0])
    for k in (1, 2, 3, 10):
        assert dr.op_matmuls(dr.OP_INV_ROOT_CN, k) == oracle.cn_inv_root(A, s, k)[2]
        assert dr.op_matmuls(dr.OP_INV_ROOT_NDB, k) == oracle.ndb_inv_root(A, s, k)[2]
    for d in (1, 2, 3, 8, 16, 32):
        assert dr.op_matmuls(dr.OP_INV_ROOT_CHEB, d) == oracle.cheb_inv_root(A, s, d, 0.01, 1.05)[1]
    assert dr.op_matmuls(dr.OP_INV_ROOT_CN, 10) == 36
    assert dr.op_matmuls(dr.OP_INV_ROOT_NDB, 10) == 54


def test_workspace_sizes():
    dr = library()
    b = 1024
    mat = b * b
    assert dr.workspace_size(dr.OP_INV_ROOT_CN, 10, b, dr.FP16, 10) >= 7 * 10 * mat * 2
    assert dr.workspace_size(dr.OP_INV_ROOT_CN, 10, b, dr.FP32_3XTF32, 10) >= 7 * 10 * mat * 8
    assert dr.workspace_size(dr.OP_INV_ROOT_NDB, 10, b, dr.TF32, 10) >= 6 * 10 * mat * 4
    assert dr.workspace_size(dr.OP_INV_ROOT_CHEB, 10, b, dr.BF16, 16) >= 4 * 10 * mat * 2
    assert dr.workspace_size(dr.OP_ACCUMULATE, 10, b, dr.BF16, 0) == 0
    assert dr.workspace_size(dr.OP_SPECTRAL_SCALE, 10, b, 0, 32) >= 2 * 10 * b * 32 * 4
    # Half-precision power modes also hold a 16-bit copy of A.
    for prec in (dr.FP16, dr.BF16):
        assert dr.workspace_size(dr.OP_SPECTRAL_SCALE, 10, b, prec, 32) >= (
            10 * mat * 2 + 2 * 10 * b * 32 * 2)


def test_bad_arguments_rejected_on_host():
    dr = library()
    lib = dr.load_library()
    null = ctypes.c_void_p(0)
    bad = ctypes.c_void_p(8)  # misaligned, never dereferenced
    sz = ctypes.c_size_t(0)
    # B not a multiple of 128 / out of range / bad precision.
    assert lib.dash_workspace_size(2, 4, 100, 0, 10, ctypes.byref(sz)) == 1
    assert lib.dash_workspace_size(2, 4, 4096, 0, 10, ctypes.byref(sz)) == 1
    assert lib.dash_workspace_size(2, 4, 256, 9, 10, ctypes.byref(sz)) == 1
    assert lib.inv_root_cn(null, 0.0, null, 4, 100, 10, 0, null, null, null, 0, null) == 1
    assert lib.inv_root_cn(null, 0.0, null, 4, 128, 0, 0, null, null, null, 0, null) == 1
    assert lib.inv_root_ndb(null, 0.0, null, 4, 128, 10, 7, null, null, null, 0, null) == 1
    assert lib.inv_root_cheb(null, 0.0, null, 4, 128, 0, 0.01, 1.0, 0, null, null, 0, null) == 1
    assert lib.inv_root_cheb(null, 0.0, null, 4, 128, 8, 1.0, 0.5, 0, null, null, 0, null) == 1
    # Misaligned pointers.
    assert lib.inv_root_cn(bad, 0.0, bad, 4, 128, 10, 0, bad, null, null, 0, null) == 1
    assert lib.dash_gemm(bad, null, 0, bad, null, 0, 2, 128, 1, bad, null) == 1
    # Null workspace where one is required.
    assert lib.spectral_scale(ctypes.c_void_p(256), 0.0, 2, 128, 0, 32, 10,
                              ctypes.c_void_p(512), ctypes.c_void_p(1024), null, 0, null) == 1
    # Unknown scale mode; a half-precision power mode without start vectors.
    assert lib.spectral_scale(ctypes.c_void_p(256), 0.0, 2, 128, 4, 32, 10,
                              ctypes.c_void_p(512), ctypes.c_void_p(1024),
                              ctypes.c_void_p(2048), 1 << 20, null) == 1
    for mode in (dr.SCALE_POWER_F16, dr.SCALE_POWER_BF16):
        assert lib.spectral_scale(ctypes.c_void_p(256), 0.0, 2, 128, mode, 32, 10, null,
                                  ctypes.c_void_p(1024), ctypes.c_void_p(2048), 1 << 20,
                                  null) == 1
    # Block packing: ld < cols, unknown dtype, B out of range; update without W.
    assert lib.pack_blocks(ctypes.c_void_p(256), 0, 4, 8, 7, 128, ctypes.c_void_p(512), null,
                           null, null) == 1
    assert lib.pack_blocks(ctypes.c_void_p(256), 9, 4, 8, 8, 128, ctypes.c_void_p(512), null,
                           null, null) == 1
    assert lib.unpack_blocks(ctypes.c_void_p(256), 1, 4, 8, 8, 100, ctypes.c_void_p(512),
                             null) == 1
    assert lib.pack_blocks(null, 0, 0, 8, 8, 128, null, null, null, null) == 0  # empty
    assert lib.precondition_update(ctypes.c_void_p(256), 1, ctypes.c_void_p(512), 2, 128, 1,
                                   ctypes.c_float(0.1), null, null, ctypes.c_void_p(1024),
                                   1 << 20, null) == 1
    assert lib.precondition_update(ctypes.c_void_p(256), 1, ctypes.c_void_p(512), 2, 128, 1,
                                   ctypes.c_float(float("nan")), ctypes.c_void_p(768), null,
                                   ctypes.c_void_p(1024), 1 << 20, null) == 1
    assert lib.precondition_apply(ctypes.c_void_p(256), 1, ctypes.c_void_p(512), 2, 128, 1,
                                  null, ctypes.c_void_p(1024), 1 << 20, null) == 1
    # beta outside [0, 1].
    assert lib.shampoo_accumulate(ctypes.c_void_p(256), 1, 2, 128, ctypes.c_float(1.5),
                                  ctypes.c_void_p(512), null, null, null, 0, null) == 1
    # N == 0 is a no-op.
    assert lib.inv_root_cn(null, 0.0, null, 0, 128, 10, 0, null, null, null, 0, null) == 0
    assert lib.dash_gemm(null, null, 0, null, null, 0, 0, 128, 1, null, null) == 0


def test_root_tf32_flag_checked():
    """DASH_ROOT_TF32 is accepted by the root solvers and, with TF32 only, by apply;
    any other flag bit or combination is an argument error found on the host."""
    dr = library()
    lib = dr.load_library()
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: every call fails before a launch
    f = dr.ROOT_TF32
    for prec in (dr.FP16 | f, dr.TF32 | f, dr.FP32_3XTF32 | f):  # too small, not invalid
        assert lib.inv_root_cn(p, 0.0, p, 4, 1024, 10, prec, p, None, p, 4096, None) == 4
        assert lib.inv_root_ndb(p, 0.0, p, 4, 1024, 10, prec, p, None, p, 4096, None) == 4
    assert lib.precondition_apply(p, 1, p, 4, 1024, dr.TF32 | f, p, p, 4096, None) == 4
    for prec in (dr.FP16 | 0x200, dr.FP16 | f | 0x200, 4 | f):
        assert lib.inv_root_cn(p, 0.0, p, 4, 1024, 10, prec, p, None, p, 4096, None) == 1
        assert lib.inv_root_cheb(p, 0.0, p, 4, 1024, 8, ctypes.c_double(0.01),
                                 ctypes.c_double(1.05), prec, p, p, 4096, None) == 1
    for prec in (dr.FP16 | f, dr.BF16 | f, dr.FP32_3XTF32 | f, dr.TF32 | 0x200):
        assert lib.precondition_apply(p, 1, p, 4, 1024, prec, p, p, 4096, None) == 1
    assert dr._prec("tf32+root_tf32") == dr.TF32 | f
    with pytest.raises(ValueError):
        dr._prec("tf32+fast")
    assert (dr.workspace_size(dr.OP_INV_ROOT_CN, 4, 1024, dr.FP16 | f, 10)
            == dr.workspace_size(dr.OP_INV_ROOT_CN, 4, 1024, dr.FP16, 10))


def test_workspace_too_small_reported():
    dr = library()
    lib = dr.load_library()
    p = ctypes.c_void_p(1 << 20)  # 256-aligned, never dereferenced: fails before any launch
    # Room for the per-call arrays but not for one block's iterates.
    assert lib.inv_root_cn(p, 0.0, p, 4, 1024, 10, 0, p, None, p, 4096, None) == 4
    assert lib.inv_root_ndb(p, 0.0, p, 4, 1024, 10, 2, p, None, p, 4096, None) == 4
    assert lib.precondition_apply(p, 1, p, 4, 1024, 0, p, p, 4096, None) == 4
    # Half-precision power: one block's 16-bit copy (2 MiB at B = 1024) does not fit.
    assert lib.spectral_scale(p, 0.0, 4, 1024, dr.SCALE_POWER_F16, 32, 10, p, p, p, 4096,
                              None) == 4


def test_binding_shape_checks():
    """The binding rejects sizes the kernels would index past, before any call."""
    import torch

    dr = library()
    t = torch.empty((3, 4, 4))
    assert dr._shape(t, (3, 4, 4), "t") is t
    with pytest.raises(ValueError, match="must have shape"):
        dr._shape(t, (2, 4, 4), "t")
    assert dr._blocks3(t, "t") == (3, 4)
    for bad in (torch.empty((3, 4, 5)), torch.empty((4, 4))):
        with pytest.raises(ValueError, match="stack"):
            dr._blocks3(bad, "t")
    assert dr._nbytes(None) == 0
    assert dr._nbytes(torch.empty(10, dtype=torch.float32)) == 40
    assert dr._nbytes(torch.empty(10, dtype=torch.uint8)) == 10


def test_binding_requires_cuda_tensors():
    import torch

    dr = library()
    G = torch.zeros((2, 128, 128), dtype=torch.bfloat16)
    F = torch.zeros((4, 128, 128))
    with pytest.raises(TypeError, match="CUDA"):
        dr.shampoo_accumulate(G, F, 0.9)
    with pytest.raises(TypeError, match="CUDA"):
        dr.inv_root_cn(F, torch.ones(4), 3)
    with pytest.raises(TypeError, match="CUDA"):
        dr.gemm(F, F)


@pytest.mark.parametrize("d,lo,hi", [(1, 0.01, 1.05), (8, 0.01, 1.05), (16, 0.05, 2.0),
                                     (32, 0.01, 1.05), (64, 1e-3, 1.0)])
def test_library_chebyshev_coefficients_match_oracle(d, lo, hi):
    """The coefficients inv_root_cheb computes on the host, against the oracle's
    (itself pinned to numpy's chebinterpolate)."""
    import numpy as np

    dr = library()
    got = np.array(dr.cheb_coeffs(d, lo, hi))
    want = oracle.cheb_coeffs(d, lo, hi)
    assert got.shape == want.shape
    assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want))


def test_chebyshev_coefficients_bad_arguments():
    dr = library()
    for args in ((0, 0.01, 1.05), (65, 0.01, 1.05), (8, 0.0, 1.0), (8, 1.0, 0.5),
                 (8, 0.01, float("inf"))):
        with pytest.raises(dr.DashError):
            dr.cheb_coeffs(*args)


def test_library_tier_selection_matches_oracle():
    """The library's host-side tier rule against the oracle's, on float32 estimates
    including the edge cases (a gate boundary, lambda_min <= 0, NaN, inf)."""
    import numpy as np

    dr = library()
    rng = np.random.default_rng(40)
    lmax = rng.uniform(0.5, 2.0, 200).astype(np.float32)
    lmin = (lmax / 10.0 ** rng.uniform(0, 7, 200)).astype(np.float32)
    t0 = oracle.DEFAULT_TIERS[0]
    edge = 4.0 * t0["gate"] / t0["u"]
    extra_max = np.array([1.0, 1.0, 1.0, 1.0, np.nan, np.inf, 1.0, -1.0, 0.0],
                         dtype=np.float32)
    extra_min = np.array([1.0 / edge, 0.0, -1.0, np.nan, 0.5, 0.5, 1e-30, 0.5, 0.5],
                         dtype=np.float32)
    lmax = np.concatenate([lmax, extra_max])
    lmin = np.concatenate([lmin, extra_min])
    got = dr.select_tiers(lmax, lmin, oracle.DEFAULT_TIERS)
    want = oracle.select_tiers(oracle.condition_estimate(lmax.astype(np.float64),
                                                         lmin.astype(np.float64)))
    assert got == want.tolist()
    assert set(got[:200]) == {0, 1}
    # A block with no usable lambda_max estimate (negative or zero) goes to the
    # last, most accurate tier, like one with no resolved lambda_min.
    assert got[-2:] == [len(oracle.DEFAULT_TIERS) - 1] * 2
    tiers3 = [dict(t0), {"solver": "ndb", "prec": "tf32", "iters": 12, "u": 2.0 ** -24,
                         "gate": 1.0}, dict(oracle.DEFAULT_TIERS[1])]
    got3 = dr.select_tiers(lmax, lmin, tiers3)
    assert got3 == oracle.select_tiers(oracle.condition_estimate(
        lmax.astype(np.float64), lmin.astype(np.float64)), tiers3).tolist()
    assert dr.select_tiers([], [], tiers3) == []


def test_library_tier_selection_bad_tiers():
    dr = library()
    good = dict(oracle.DEFAULT_TIERS[0])
    for bad in ({"iters": 0}, {"u": 0.0}, {"gate": -1.0}, {"prec": 9}):
        t = dict(good)
        t.update(bad)
        with pytest.raises(dr.DashError):
            dr.select_tiers([1.0], [0.5], [t])


def test_library_default_tiers_are_the_oracles():
    """The binding's default tiers (used by bench.py and inv_root_auto callers) and
    the oracle's are written separately; they must agree."""
    import matrix_inverse_roots_gb300 as dr

    assert [dict(t) for t in dr.DEFAULT_TIERS] == [dict(t) for t in oracle.DEFAULT_TIERS]
