"""spectral_scale_noalloc, the scaling entry point for callers that cannot
allocate device memory, against the workspace-taking spectral_scale.

Kept in its own file, collected after every other test file, so that a run
stopping at the first failure has already run everything else.  It must pass
both alone in a fresh process (the first call then does the per-device lookup
of the built-in scratch) and after the other tests (the shared scratch then
holds leftovers of earlier calls)."""

import ctypes

import numpy as np
import pytest
import torch

import synth
from tests.helpers import library, require_gpu, to64

pytestmark = pytest.mark.gpu

LAMBDA_TOL = 1e-5  # same relative tolerance as the power-iteration parity tests


def call_noalloc(lib, A, mode, V0, iters, ridge, out):
    n, b, _ = A.shape
    nv = 0 if V0 is None else V0.shape[2]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.spectral_scale_noalloc(
        ctypes.c_void_p(A.data_ptr()), ctypes.c_float(ridge), n, b, mode, nv, iters,
        None if V0 is None else ctypes.c_void_p(V0.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), stream)


def test_noalloc_matches_workspace_entry_point_twice():
    require_gpu()
    dr = library()
    lib = dr.load_library()
    cases = [
        (synth.wishart(16, 1024, seed=31, device="cuda"), 1e-3, 10, 32),
        (synth.wishart(40, 256, seed=32, device="cuda"), 0.0, 7, 13),
    ]
    for A, ridge, iters, nv in cases:  # two calls in a row, different shapes
        V0 = synth.start_vectors(A.shape[0], A.shape[1], nv, seed=33, device="cuda")
        ref = dr.spectral_scale(A, dr.SCALE_POWER, V0, iters, ridge=ridge)
        out = torch.full((A.shape[0],), float("nan"), device="cuda")
        assert call_noalloc(lib, A, dr.SCALE_POWER, V0, iters, ridge, out) == 0
        torch.cuda.synchronize()
        assert dr.device_status() == 0
        r, o = to64(ref), to64(out)
        assert np.all(np.isfinite(o))
        assert np.max(np.abs(o - r) / r) < LAMBDA_TOL
        # Frobenius mode through the same scratch.
        ref_f = dr.spectral_scale(A, dr.SCALE_FROBENIUS, ridge=ridge)
        out_f = torch.full((A.shape[0],), float("nan"), device="cuda")
        assert call_noalloc(lib, A, dr.SCALE_FROBENIUS, None, 0, ridge, out_f) == 0
        torch.cuda.synchronize()
        assert np.max(np.abs(to64(out_f) - to64(ref_f)) / to64(ref_f)) < LAMBDA_TOL


def test_noalloc_refuses_stacks_beyond_its_scratch():
    require_gpu()
    dr = library()
    lib = dr.load_library()
    # 128 blocks of 1024^2 with 32 vectors need more than the 32 MiB scratch.
    A = torch.empty((128, 1024, 1024), device="cuda")
    V0 = torch.empty((128, 1024, 32), device="cuda")
    out = torch.empty(128, device="cuda")
    assert call_noalloc(lib, A, dr.SCALE_POWER, V0, 3, 0.0, out) == 4  # WORKSPACE_TOO_SMALL
    assert dr.NOALLOC_SCRATCH_BYTES == 32 * 1024 * 1024
