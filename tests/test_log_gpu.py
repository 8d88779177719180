"""GPU parity of mg_log_scan_fwd against the float64 oracle."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from linear_recurrence_scans_gb300 import workloads as wl
from parity import TOL_F32, log_fwd_errors

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check(mg, lc, lv, tol=TOL_F32):
    lcd, lvd = lc.to(DEV), lv.to(DEV)
    h = mg.parallel_scan_log_fwd(lcd, lvd, out=torch.full_like(lcd, float("nan")))
    assert not torch.isnan(h).any()
    errs = log_fwd_errors(lc, lv, h)
    assert max(errs.values()) <= tol, errs
    mg.workspace_status()
    return errs


@pytest.mark.parametrize("shape", [(1, 1, 4), (2, 7, 4), (3, 513, 300), (2, 700, 37),
                                   (1, 5000, 8)])
def test_mingru_log_shapes(cuda_lib, shape):
    lc, lv = wl.mingru_log(*shape, seed=11)
    _check(cuda_lib, lc, lv)


def test_mingru_log_16x2048x2048_full(cuda_lib):
    lc, lv = wl.mingru_log(16, 2048, 2048, seed=0)
    print("mingru_log_16x2048x2048", _check(cuda_lib, lc, lv))


def test_zero_terms_give_zero_not_nan(cuda_lib):
    """-inf log inputs are zero coefficients / values: h = 0 where every term
    vanishes, and the recurrence restarts cleanly afterwards."""
    B, T, D = 2, 300, 8
    lc, lv = wl.mingru_log(B, T, D, seed=12)
    lc[0, 50:60] = -math.inf          # coefficient zero: forget the past
    lv[0, 51:61] = -math.inf          # and no new value -> h = 0 on 51..60 (steps)
    lv[1, 0] = -math.inf              # h_0 = 0
    lc[1, :, :4] = -math.inf          # every coefficient zero on 4 channels
    lv[1, 1:100, :4] = -math.inf      # ... and no values for 99 steps -> h = 0
    _check(cuda_lib, lc, lv)
    h = cuda_lib.parallel_scan_log_fwd(lc.to(DEV), lv.to(DEV)).cpu()
    assert torch.all(h[0, 50:60] == 0)
    assert torch.all(h[1, :99, :4] == 0)


def test_wide_dynamic_range(cuda_lib):
    """Log values far outside float32's exp range on the way (the running
    coefficient product underflows in linear float32) while h stays finite."""
    B, T, D = 1, 600, 16
    g = torch.Generator().manual_seed(13)
    lc = -torch.rand(B, T, D, generator=g) * 3.0
    lv = torch.randn(B, T + 1, D, generator=g) * 2.0
    lv[:, 0] = 100.0    # h_0 = e^100 is beyond float32 range ...
    lc[:, :5] = -20.0   # ... decayed by e^-100 within five steps
    _check(cuda_lib, lc, lv)


def test_bitwise_reproducible(cuda_lib):
    lc, lv = wl.mingru_log(4, 2048, 512, seed=14, device=DEV)
    h1 = cuda_lib.parallel_scan_log_fwd(lc, lv)
    h2 = cuda_lib.parallel_scan_log_fwd(lc, lv)
    assert torch.equal(h1, h2)
