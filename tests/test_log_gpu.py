"""GPU parity of mg_log_scan_fwd and its adjoint mg_log_scan_bwd against the
float64 oracle."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from linear_recurrence_scans_gb300 import workloads as wl
from parity import TOL_F32, log_bwd_errors, log_fwd_errors

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


# ------------------------------------------------------------- the adjoint

def _check_bwd(mg, lc, lv, gh, tol=TOL_F32):
    """GPU adjoint with the oracle's forward h (rounded to float32) as input;
    outputs start as NaN so an unwritten element fails."""
    import oracle
    h32 = torch.from_numpy(oracle.log_scan_fwd(lc, lv)).float()
    lcd, lvd = lc.to(DEV), lv.to(DEV)
    dlc, dlv = mg.parallel_scan_log_bwd(
        lcd, lvd, h32.to(DEV), gh.to(DEV),
        out=(torch.full_like(lcd, float("nan")), torch.full_like(lvd, float("nan"))))
    assert not torch.isnan(dlc).any() and not torch.isnan(dlv).any()
    errs = log_bwd_errors(lc, lv, gh, dlc, dlv)
    assert max(errs.values()) <= tol, errs
    mg.workspace_status()
    return errs


@pytest.mark.parametrize("shape", [(1, 1, 4), (2, 7, 4), (3, 513, 300), (2, 700, 37),
                                   (1, 5000, 8), (2, 1000, 512)])
def test_log_bwd_shapes(cuda_lib, shape):
    lc, lv = wl.mingru_log(*shape, seed=21)
    g = torch.Generator().manual_seed(22)
    gh = torch.randn(lc.shape, generator=g)
    _check_bwd(cuda_lib, lc, lv, gh)


def test_log_bwd_16x2048x2048_full(cuda_lib):
    lc, lv = wl.mingru_log(16, 2048, 2048, seed=0)
    gh = torch.randn(lc.shape, generator=torch.Generator().manual_seed(1))
    print("mingru_log_bwd_16x2048x2048", _check_bwd(cuda_lib, lc, lv, gh))


def test_log_bwd_zero_terms(cuda_lib):
    """-inf coefficients (a forgotten past) and -inf values (zero inputs)."""
    B, T, D = 2, 300, 8
    lc, lv = wl.mingru_log(B, T, D, seed=23)
    lc[0, 50:60] = -math.inf
    lv[0, 51:61] = -math.inf
    lv[1, 0] = -math.inf
    gh = torch.randn(lc.shape, generator=torch.Generator().manual_seed(24))
    _check_bwd(cuda_lib, lc, lv, gh)


def test_log_bwd_t0_zero_fills(cuda_lib):
    mg = cuda_lib
    lc = torch.zeros(2, 0, 4, device=DEV)
    lv = torch.randn(2, 1, 4, device=DEV)
    dlc, dlv = mg.parallel_scan_log_bwd(lc, lv, lc, lc, out=(None, torch.full_like(lv, float("nan"))))
    assert dlc.shape == (2, 0, 4) and torch.all(dlv == 0)


def test_log_bwd_bitwise_reproducible(cuda_lib):
    lc, lv = wl.mingru_log(4, 2048, 512, seed=25, device=DEV)
    h = cuda_lib.parallel_scan_log_fwd(lc, lv)
    gh = torch.randn(lc.shape, device=DEV)
    r1 = cuda_lib.parallel_scan_log_bwd(lc, lv, h, gh)
    r2 = cuda_lib.parallel_scan_log_bwd(lc, lv, h, gh)
    assert torch.equal(r1[0], r2[0]) and torch.equal(r1[1], r2[1])
