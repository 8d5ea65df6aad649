"""spectral_scale_noalloc, the scaling entry point for callers that cannot
allocate device memory, against the workspace-taking spectral_scale and the
float64 oracle.

Kept in its own file, collected after every other test file, so that a run
stopping at the first failure has already run everything else.  It must pass
both alone in a fresh process (the first call then does the per-device lookup
of the built-in scratch) and after the other tests (the shared scratch then
holds leftovers of earlier calls)."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import library, require_gpu, to64

pytestmark = pytest.mark.gpu

LAMBDA_TOL = 1e-5     # same relative tolerance as the power-iteration parity tests
HALF_TOL = 4 * 2.0 ** -11  # half-precision iteration against the oracle on the fp16 copy
WORKSPACE_TOO_SMALL = 4


def call_noalloc(lib, A, mode, V0, iters, ridge, out):
    n, b, _ = A.shape
    nv = 0 if V0 is None else V0.shape[2]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.spectral_scale_noalloc(
        ctypes.c_void_p(A.data_ptr()), ctypes.c_float(ridge), n, b, mode, nv, iters,
        None if V0 is None else ctypes.c_void_p(V0.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), stream)


def rel(a, b):
    a, b = to64(a) if torch.is_tensor(a) else a, to64(b) if torch.is_tensor(b) else b
    return float(np.max(np.abs(a - b) / np.abs(b)))


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
        assert np.all(np.isfinite(to64(out)))
        assert rel(out, ref) < LAMBDA_TOL
        # and the float64 oracle on the same inputs
        want = oracle.power_lambda(to64(A), to64(V0), iters, ridge=ridge)
        assert rel(out, want) < LAMBDA_TOL
        # Frobenius mode through the same scratch.
        ref_f = dr.spectral_scale(A, dr.SCALE_FROBENIUS, ridge=ridge)
        out_f = torch.full((A.shape[0],), float("nan"), device="cuda")
        assert call_noalloc(lib, A, dr.SCALE_FROBENIUS, None, 0, ridge, out_f) == 0
        torch.cuda.synchronize()
        assert rel(out_f, ref_f) < LAMBDA_TOL
        assert rel(out_f, oracle.frobenius_norm(to64(A), ridge=ridge)) < LAMBDA_TOL


def test_noalloc_half_precision_mode_twice():
    # The fp16 iteration keeps its 16-bit copy of every block and the per-block
    # power-of-two scale in the shared scratch too.
    require_gpu()
    dr = library()
    lib = dr.load_library()
    cases = [(synth.wishart(15, 1024, seed=41, device="cuda"), 1e-6, 10, 32),   # the limit
             (synth.wishart(24, 512, seed=42, device="cuda") * 1e-4, 0.0, 6, 32)]
    for A, ridge, iters, nv in cases:
        V0 = synth.start_vectors(A.shape[0], A.shape[1], nv, seed=43, device="cuda")
        ref = dr.spectral_scale(A, dr.SCALE_POWER_F16, V0, iters, ridge=ridge)
        out = torch.full((A.shape[0],), float("nan"), device="cuda")
        assert call_noalloc(lib, A, dr.SCALE_POWER_F16, V0, iters, ridge, out) == 0
        torch.cuda.synchronize()
        assert dr.device_status() == 0
        assert rel(out, ref) < LAMBDA_TOL
        # The oracle on the 16-bit copy the iteration reads (sigma is a power of two,
        # so rounding A to fp16 and rounding sigma A are the same up to scale).
        sig = 2.0 ** -np.floor(np.log2(np.maximum(to64(A).diagonal(0, 1, 2).max(1), ridge)) + 1)
        Ah = (A * torch.tensor(sig, device="cuda", dtype=torch.float32)[:, None, None]).half()
        want = np.array([oracle.power_lambda(to64(Ah[k:k + 1]), to64(V0[k:k + 1]), iters,
                                             ridge=ridge * sig[k])[0] / sig[k]
                         for k in range(A.shape[0])])
        assert rel(out, want) < HALF_TOL


def test_noalloc_refuses_stacks_beyond_its_scratch():
    require_gpu()
    dr = library()
    lib = dr.load_library()
    assert dr.NOALLOC_SCRATCH_BYTES == 32 * 1024 * 1024
    # 128 blocks of 1024^2 with 32 vectors need more than the 32 MiB scratch,
    # and so do 16 blocks in a half-precision mode (their 16-bit copies).
    for n, mode in ((128, dr.SCALE_POWER), (16, dr.SCALE_POWER_F16), (16, dr.SCALE_POWER_BF16)):
        A = torch.empty((n, 1024, 1024), device="cuda")
        V0 = torch.empty((n, 1024, 32), device="cuda")
        out = torch.empty(n, device="cuda")
        assert call_noalloc(lib, A, mode, V0, 3, 0.0, out) == WORKSPACE_TOO_SMALL
