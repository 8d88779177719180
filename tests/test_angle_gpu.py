"""GPU parity of the angle-fused scan (mg_angle_scan_fwd / mg_angle_scan_bwd)
against the float64 oracle's reading of it, through the C ABI (via the
Python binding).  Outputs start as NaN so an unwritten element fails.

Tolerance.  The states and their gradients (h, db, dh0) are measured
against the RMS over the state's k coordinates (rotations are stable
normwise, not entrywise, as for the affine outputs); dtheta, dscale and
dgamma against their Cauchy-Schwarz magnitude |factor| |lam_t| |h_{t-1}|."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from linear_recurrence_scans_gb300 import workloads as wl
from parity import TOL_F32, scaled_error

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _np(x):
    return x.detach().to("cpu", torch.float64).numpy()


def _rms_last(x, axis=-1):
    x = np.asarray(x, dtype=np.float64)
    return np.broadcast_to(np.sqrt(np.mean(x * x, axis=axis, keepdims=True)), x.shape)


def _case(mg, B, T, n, R, k, seed, has_scale=1, has_decay=1):
    import oracle
    th, sc, ga, b, h0, perm, sgn, p2p, go = wl.angle_inputs(B, T, n, R, k, seed=seed)
    nan = lambda shape: torch.full(tuple(shape), float("nan"), device=DEV)  # noqa: E731
    h = mg.angle_scan_fwd(th.to(DEV), sc.to(DEV), ga.to(DEV), b.to(DEV), h0.to(DEV), perm, sgn,
                          p2p, has_scale=has_scale, has_decay=has_decay, out=nan(b.shape))
    rh = oracle.angle_scan_fwd(th, sc, ga, b, h0, perm, sgn, has_scale, has_decay)
    errs = {"h": scaled_error(_np(h), rh, _rms_last(rh))}
    assert max(errs.values()) <= TOL_F32, errs
    h32 = torch.from_numpy(rh).float()
    outs = (nan(th.shape), nan(sc.shape), nan(ga.shape), nan(b.shape), nan(h0.shape))
    got = mg.angle_scan_bwd(th.to(DEV), sc.to(DEV), ga.to(DEV), h0.to(DEV), h32.to(DEV),
                            go.to(DEV), perm, sgn, p2p, has_scale=has_scale, has_decay=has_decay,
                            out=outs)
    ref = oracle.angle_scan_bwd(th, sc, ga, h0, h32, go, perm, sgn, has_scale, has_decay)
    # scales: each of dtheta, dscale, dgamma at step t is an inner product of
    # the gradient carried back from lam_t = db_t with a vector that the
    # (norm-preserving for sgn = +-1) layers make from h_{t-1}, so by
    # Cauchy-Schwarz its natural magnitude is |f| |lam_t| |h_{t-1}| with f the
    # scalar factor in front (s g, g or s); db, dh0 against the state RMS
    lam = np.linalg.norm(ref[3], axis=-1)                              # (B,T,n)
    hp = np.concatenate([_np(h0)[:, None], rh[:, :-1]], axis=1)
    hn = np.linalg.norm(hp, axis=-1)
    s_ = _np(sc) if has_scale else np.ones_like(lam)
    g_ = _np(ga) if has_decay else np.ones_like(lam)
    S = [np.broadcast_to((np.abs(s_ * g_) * lam * hn)[..., None, None], ref[0].shape),
         np.abs(g_) * lam * hn, np.abs(s_) * lam * hn,
         _rms_last(ref[3]), _rms_last(ref[4])]
    for name, g, r, s in zip(("dtheta", "dscale", "dgamma", "db", "dh0"), got, ref, S):
        errs[name] = scaled_error(_np(g), r, s)
    assert max(errs.values()) <= TOL_F32, errs
    if not has_scale:
        assert not got[1].any()
    if not has_decay:
        assert not got[2].any()
    return errs


@pytest.mark.parametrize("k,R", [(2, 1), (4, 3), (8, 2), (16, 4), (32, 8)])
def test_angle_shapes(cuda_lib, k, R):
    _case(cuda_lib, 2, 300, 5, R, k, seed=61)


@pytest.mark.parametrize("flags", [(1, 0), (0, 1), (0, 0)])
def test_angle_flags(cuda_lib, flags):
    _case(cuda_lib, 2, 200, 3, 2, 8, seed=62, has_scale=flags[0], has_decay=flags[1])


def test_angle_many_sequences_long(cuda_lib):
    """Several warps and blocks, a ragged last block (B*n*k not a multiple of
    the block), T not a multiple of the steps loaded ahead."""
    print(_case(cuda_lib, 3, 2051, 37, 4, 16, seed=63))


def test_angle_rejects_bad_constants(cuda_lib):
    mg = cuda_lib
    th, sc, ga, b, h0, perm, sgn, p2p, _ = wl.angle_inputs(1, 4, 2, 2, 4, seed=64, device=DEV,
                                                            grads=False)
    bad = perm.clone()
    bad[0, 0] = bad[0, 1]
    with pytest.raises(mg.MgScanError):
        mg.angle_scan_fwd(th, sc, ga, b, h0, bad, sgn)
    with pytest.raises(mg.MgScanError):
        mg.angle_scan_fwd(th, sc, ga, b, h0, perm, sgn, torch.flip(p2p, [1]))
