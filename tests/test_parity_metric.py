"""CPU checks of the parity metric itself (no GPU)."""
from __future__ import annotations

import numpy as np
import torch

from parity import affine_bwd_errors, affine_fwd_errors, linear_bwd_errors, linear_fwd_errors, scaled_error


def test_scaled_error_basics():
    r = np.array([1.0, -2.0, 0.0])
    assert scaled_error(r, r) == 0.0
    assert np.isclose(scaled_error(r * (1 + 1e-5), r), 1e-5)
    # a zero reference is measured against its scale S, not against |r| = 0
    assert np.isclose(scaled_error(np.array([1e-6]), np.array([0.0]), np.array([1.0])), 1e-6)
    assert scaled_error(np.array([np.nan]), np.array([1.0])) == float("inf")


def _perturbed(x, rel, seed):
    g = torch.Generator().manual_seed(seed)
    return x * (1 + rel * torch.randn(x.shape, generator=g, dtype=torch.float64))


def test_k1_affine_metric_matches_the_linear_one():
    """With k = v = 1 the affine scan is the linear recurrence; the affine
    metric then uses the same componentwise scale, so a perturbed result
    scores like it does under the linear metric (the product outputs get
    |r| + |r| as denominator there instead of |r|, hence the factor 2)."""
    g = torch.Generator().manual_seed(5)
    a = torch.rand(2, 300, 4, generator=g, dtype=torch.float64) * 1.6 - 0.8
    b = torch.randn(2, 300, 4, generator=g, dtype=torch.float64)
    gA = torch.randn(a.shape, generator=g, dtype=torch.float64)
    gB = torch.randn(a.shape, generator=g, dtype=torch.float64)
    import oracle
    rA, rBc = (torch.from_numpy(x) for x in oracle.linear_scan_fwd(a, b))
    A, Bc = _perturbed(rA, 1e-6, 1), _perturbed(rBc, 1e-6, 2)
    lin = linear_fwd_errors(a, b, A, Bc)
    aff = affine_fwd_errors(a[..., None, None], b[..., None, None], A[..., None, None], Bc[..., None, None])
    assert np.isclose(aff["Bbar"], lin["Bc"])
    assert np.isclose(2 * aff["Abar"], lin["A"], rtol=1e-6)
    rda, rdb = (torch.from_numpy(x) for x in oracle.linear_scan_bwd(a, rA, rBc, gA, gB))
    da, db = _perturbed(rda, 1e-6, 3), _perturbed(rdb, 1e-6, 4)
    lin_b = linear_bwd_errors(a, rA, rBc, gA, gB, da, db)
    e = lambda x: x[..., None, None]  # noqa: E731
    aff_b = affine_bwd_errors(e(a), e(rA), e(rBc), e(gA), e(gB), e(da), e(db))
    assert np.isclose(aff_b["dA"], lin_b["da"]) and np.isclose(aff_b["dB"], lin_b["db"])


def test_k2_affine_metric_uses_the_block_scale():
    """For k >= 2 an element near zero inside a block of normal size is
    measured against the block's RMS."""
    g = torch.Generator().manual_seed(6)
    A = torch.randn(1, 5, 1, 2, 2, generator=g, dtype=torch.float64) * 0.5
    Bm = torch.randn(1, 5, 1, 2, 2, generator=g, dtype=torch.float64)
    import oracle
    rAbar, rBbar = (torch.from_numpy(x) for x in oracle.affine_scan_fwd(A, Bm))
    Bbar = rBbar.clone()
    Bbar[0, 2, 0, 0, 0] += 1e-7 * float(rBbar[0, 2, 0].pow(2).mean().sqrt())
    errs = affine_fwd_errors(A, Bm, rAbar, Bbar)
    assert errs["Abar"] == 0.0 and errs["Bbar"] <= 1e-7
