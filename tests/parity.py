"""The parity metric shared by the GPU-vs-oracle tests.

The stated bar is a maximum relative error of 1e-4 for float32 inputs and
2e-2 for bf16 inputs (fp32 accumulation).  A plain elementwise |g - r| / |r|
is undefined where r passes through zero (sums of signed terms) and
meaningless where float32 underflows while float64 does not (long running
products).  So every element is measured against its own scale:

    err_i = |g_i - r_i| / (|r_i| + rho * S_i + tau),   rho = 1, tau = 1e-30

with S_i the scale that rounding error is proportional to:

* running products of positive factors (A of the linear scan, h of the log
  scan): S = 0, i.e. pure relative error, floored at tau for underflow;
* sums of signed terms in the channel-wise linear family (Bc, da, db): S is
  the same quantity evaluated by the oracle on |inputs| -- the componentwise
  condition scale sum |terms| of a sum of products;
* matrix-valued affine outputs (Abar, Bbar, dA, dB) for k >= 2: S is the
  RMS of the k x k or k x v block at the same (b, t, n) -- products of
  matrices are stable normwise, not entrywise (the same chain with |A| in
  place of A grows without bound for orthogonal A, so the componentwise scale
  says nothing there);
* affine outputs for k = 1: the scan is then the scalar linear recurrence
  (one independent recurrence per column of B), and the 1 x 1 or 1 x v
  "block" degenerates to |r| itself; S is the componentwise scale as for the
  linear family, the oracle run on |inputs|.

A NaN or inf where the reference is finite counts as an infinite error.
"""
from __future__ import annotations

import numpy as np

RHO = 1.0
TAU = 1e-30
TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def scaled_error(g, r, S=0.0, rho: float = RHO, tau: float = TAU) -> float:
    g = np.asarray(g, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    if r.size == 0:
        return 0.0
    bad = ~np.isfinite(g) & np.isfinite(r)
    if bad.any():
        return float("inf")
    den = np.abs(r) + rho * np.asarray(S, dtype=np.float64) + tau
    return float(np.max(np.abs(g - r) / den))


def block_rms(x: np.ndarray) -> np.ndarray:
    """RMS over the last two (matrix) axes, broadcast back to x's shape."""
    x = np.asarray(x, dtype=np.float64)
    rms = np.sqrt(np.mean(x * x, axis=(-2, -1), keepdims=True))
    return np.broadcast_to(rms, x.shape)


def normwise(g, r) -> float:
    """||g - r||_2 / ||r||_2, reported alongside, never gating."""
    g = np.asarray(g, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    n = np.linalg.norm(r)
    return float(np.linalg.norm(g - r) / n) if n > 0 else float(np.linalg.norm(g))


# ------------------------------------------------------- op-level checkers
# Each compares GPU outputs (torch tensors) with the oracle run on the same
# inputs and returns {name: scaled error}.  Inputs may live on the GPU; they
# are copied to the host for the oracle.

def _np(x) -> np.ndarray:
    if isinstance(x, np.ndarray):
        return x.astype(np.float64, copy=False)
    return x.detach().to("cpu", dtype=__import__("torch").float64).numpy()


def linear_fwd_errors(a, b, A, Bc) -> dict:
    import oracle
    rA, rBc = oracle.linear_scan_fwd(a, b)
    SBc = oracle.linear_scan_fwd(np.abs(_np(a)), np.abs(_np(b)))[1]
    return {"A": scaled_error(_np(A), rA), "Bc": scaled_error(_np(Bc), rBc, SBc)}


def linear_bwd_errors(a, A, Bc, gA, gBc, da, db) -> dict:
    import oracle
    rda, rdb = oracle.linear_scan_bwd(a, A, Bc, gA, gBc)
    Sda, Sdb = oracle.linear_scan_bwd(*(np.abs(_np(x)) for x in (a, A, Bc, gA, gBc)))
    return {"da": scaled_error(_np(da), rda, Sda), "db": scaled_error(_np(db), rdb, Sdb)}


def log_fwd_errors(lc, lv, h) -> dict:
    import oracle
    return {"h": scaled_error(_np(h), oracle.log_scan_fwd(lc, lv))}


def log_bwd_errors(lc, lv, gh, dlc, dlv) -> dict:
    """The log-space adjoint's outputs are sums of signed terms (mu carries the
    sign of gh): S is the oracle on |gh|, the componentwise condition scale."""
    import oracle
    rdlc, rdlv = oracle.log_scan_bwd(lc, lv, gh)
    Sdlc, Sdlv = oracle.log_scan_bwd(lc, lv, np.abs(_np(gh)))
    return {"dlog_coeffs": scaled_error(_np(dlc), rdlc, Sdlc),
            "dlog_values": scaled_error(_np(dlv), rdlv, Sdlv)}


def affine_fwd_errors(A, Bm, Abar, Bbar) -> dict:
    import oracle
    rAbar, rBbar = oracle.affine_scan_fwd(A, Bm)
    if _np(A).shape[-1] == 1:
        SA, SB = oracle.affine_scan_fwd(np.abs(_np(A)), np.abs(_np(Bm)))
    else:
        SA, SB = block_rms(rAbar), block_rms(rBbar)
    return {"Abar": scaled_error(_np(Abar), rAbar, SA),
            "Bbar": scaled_error(_np(Bbar), rBbar, SB)}


def affine_bwd_errors(A, Abar, Bbar, gAbar, gBbar, dA, dB) -> dict:
    import oracle
    rdA, rdB = oracle.affine_scan_bwd(A, Abar, Bbar, gAbar, gBbar)
    if _np(A).shape[-1] == 1:
        SA, SB = oracle.affine_scan_bwd(*(np.abs(_np(x)) for x in (A, Abar, Bbar, gAbar, gBbar)))
    else:
        SA, SB = block_rms(rdA), block_rms(rdB)
    return {"dA": scaled_error(_np(dA), rdA, SA),
            "dB": scaled_error(_np(dB), rdB, SB)}


# ----------------------------------------------------- fused minGRU gate

def _gate_scales(x1, x2):
    """z = sigmoid(x1), 1 - z, g(x2) and |g'(x2)| in float64 (tolerance scales only)."""
    x1, x2 = _np(x1), _np(x2)
    z = 1.0 / (1.0 + np.exp(-x1))
    zc = 1.0 / (1.0 + np.exp(x1))          # 1 - z without cancellation
    s2 = 1.0 / (1.0 + np.exp(-x2))
    g = np.where(x2 >= 0, x2 + 0.5, s2)
    gp = np.where(x2 >= 0, 1.0, s2 * (1 - s2))
    return z, zc, g, gp


def mingru_fwd_errors(x1, x2, A, Bc) -> dict:
    """A is a product of positive factors (S = 0); Bc a sum of positive terms
    (S = the oracle's Bc, its own componentwise scale).  A may be None."""
    import oracle
    rA, rBc = oracle.mingru_scan_fwd(x1, x2)
    out = {"Bc": scaled_error(_np(Bc), rBc, np.abs(rBc))}
    if A is not None:
        out["A"] = scaled_error(_np(A), rA)
    return out


def mingru_bwd_errors(x1, x2, A, Bc, gA, gBc, dx1, dx2) -> dict:
    """dx1 = (db g - da) z (1 - z), dx2 = db z g': S is that expression with
    the linear adjoint's componentwise scales (the oracle on |inputs|) and
    the magnitudes of each factor.  gA, A may be None (gA = 0)."""
    import oracle
    x1n, Bcn, gBcn = _np(x1), _np(Bc), _np(gBc)
    gAn = np.zeros_like(x1n) if gA is None else _np(gA)
    An = np.ones_like(x1n) if A is None else _np(A)
    r1, r2 = oracle.mingru_scan_bwd(x1n, _np(x2), An, Bcn, gAn, gBcn)
    a, _ = oracle.mingru_gate(x1n, _np(x2))
    Sda, Sdb = oracle.linear_scan_bwd(a, np.abs(An), np.abs(Bcn), np.abs(gAn), np.abs(gBcn))
    z, zc, g, gp = _gate_scales(x1, x2)
    S1 = (Sdb * g + Sda) * z * zc
    S2 = Sdb * z * gp
    return {"dx1": scaled_error(_np(dx1), r1, S1), "dx2": scaled_error(_np(dx2), r2, S2)}
