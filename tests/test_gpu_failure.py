"""Failure detection without a GPU fault.

* A device-side wait that runs out reports DASH_ERR_TIMEOUT through
  dash_device_status and leaves the context usable (the self-test kernel waits,
  with a 50 ms limit, on a barrier nothing arrives on -- the same path every
  pipeline wait of the library takes).
* Host-side fault injection: a NaN planted in one block stays in that block;
  every other block's scale, root and residuals match a clean run to rounding
  (blocks are independent through the whole step; the power step's column sums
  use atomics, so the last bits may differ between any two runs)."""

import numpy as np
import pytest
import torch

import synth
from tests.helpers import library, rel_fro_blocks, require_gpu

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    require_gpu()
    dr = library()
    assert dr.device_status() == 0
    dr.selftest_wait_timeout(50000)
    assert dr.device_status() == 5  # DASH_ERR_TIMEOUT
    assert dr.device_status() == 0  # read-and-clear
    # The context still works.
    A = synth.wishart(2, 128, seed=3, device="cuda")
    s = dr.spectral_scale(A, dr.SCALE_FROBENIUS)
    X = dr.inv_root_cn(A, s, 4, "tf32")
    torch.cuda.synchronize()
    assert torch.isfinite(X).all()
    assert dr.device_status() == 0


@pytest.mark.parametrize("prec", ["3xtf32", "fp16"])
def test_nan_in_one_block_stays_in_that_block(prec):
    require_gpu()
    dr = library()
    n, b, bad = 6, 256, 2
    A = synth.wishart(n, b, seed=11, device="cuda")
    V0 = synth.start_vectors(n, b, 32, seed=12, device="cuda")
    lam = dr.spectral_scale(A, dr.SCALE_POWER, V0, 10)
    X, r = dr.inv_root_cn(A, lam, 6, prec, resid=True)
    A2 = A.clone()
    A2[bad, 17, 5] = float("nan")
    lam2 = dr.spectral_scale(A2, dr.SCALE_POWER, V0, 10)
    X2, r2 = dr.inv_root_cn(A2, lam2, 6, prec, resid=True)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    good = [k for k in range(n) if k != bad]
    assert torch.allclose(lam[good], lam2[good], rtol=1e-6, atol=0)
    # Run-to-run difference of the clean blocks stays at the precision's level
    # (fp16 re-rounds the scaled input when lambda moves in its last bit).
    tol = {"3xtf32": 1e-5, "fp16": 2e-3}[prec]
    d = rel_fro_blocks(X2[good].double().cpu().numpy(), X[good].double().cpu().numpy())
    assert d.max() < tol, d
    assert torch.isfinite(X2[good]).all() and torch.isfinite(r2[good]).all()
    assert not torch.isfinite(X2[bad]).all()
    assert not np.isfinite(r2[bad].cpu().numpy()).all()
