"""Pins of the float64 oracle to things other than itself.

The pages print no worked example for any scan, so the oracle is pinned to:
hand-derived golden cases (tests/golden), the O(T^2) closed forms written as
brute-force Python loops, numpy/scipy routines in the special cases where the
op reduces to one (cumsum, cumprod, logsumexp), agreement between the log-space
and linear ops, between the affine op at k = v = 1 or diagonal A and the
linear op, the explicit left-multiplied running product, the orthogonal-
product invariant, central finite differences and torch.autograd for the
adjoints.

Each pin is a function of an oracle object so that ``test_planted_mistakes``
can run the whole set against deliberately broken builds of the oracle's C
source and check that every planted mistake is caught by at least one pin.
"""
from __future__ import annotations

import functools
import json
import math
import os
import shutil
import tempfile

import numpy as np
import pytest
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- pins ------

def pin_golden_linear(orc):
    g = _golden("linear_scan_T4.json")
    a, b = np.array(g["a"]), np.array(g["b"])
    A, Bc = orc.linear_scan_fwd(a, b)
    np.testing.assert_array_equal(A, np.array(g["A"]))
    np.testing.assert_array_equal(Bc, np.array(g["Bc"]))
    da, db = orc.linear_scan_bwd(a, np.array(g["A"]), np.array(g["Bc"]),
                                 np.array(g["gA"]), np.array(g["gBc"]))
    np.testing.assert_array_equal(da, np.array(g["da"]))
    np.testing.assert_array_equal(db, np.array(g["db"]))


def pin_golden_log(orc):
    g = _golden("log_scan_T3.json")
    with np.errstate(divide="ignore"):
        for case in g["cases"]:
            lc = np.log(np.array(case["log_coeffs_exp"], dtype=np.float64))
            lv = np.log(np.array(case["log_values_exp"], dtype=np.float64))
            h = orc.log_scan_fwd(lc, lv)
            np.testing.assert_allclose(h, np.array(case["h"]), rtol=1e-14, atol=0,
                                       err_msg=case["name"])
            assert np.all(np.isfinite(h))


def pin_golden_affine(orc):
    g = _golden("affine_scan_k2.json")
    A, Bm = np.array(g["A"]), np.array(g["Bm"])
    Abar, Bbar = orc.affine_scan_fwd(A, Bm)
    np.testing.assert_array_equal(Abar, np.array(g["Abar"]))
    np.testing.assert_array_equal(Bbar, np.array(g["Bbar"]))
    dA, dB = orc.affine_scan_bwd(A, np.array(g["Abar"]), np.array(g["Bbar"]),
                                 np.array(g["gAbar"]), np.array(g["gBbar"]))
    np.testing.assert_array_equal(dA, np.array(g["dA"]))
    np.testing.assert_array_equal(dB, np.array(g["dB"]))


def _tiny_linear(seed, B=2, T=13, D=3, positive=False):
    rng = np.random.default_rng(seed)
    a = rng.uniform(0.2, 1.3, (B, T, D)) * (1 if positive else rng.choice([-1, 1], (B, T, D)))
    b = rng.normal(size=(B, T, D))
    if positive:
        b = np.abs(b) + 0.1
    return a, b


def pin_linear_closed_form(orc):
    """A_t = prod_{r<=t} a_r and h_t = sum_{s<=t} (prod_{s<r<=t} a_r) b_s, by brute force."""
    for seed in range(3):
        a, b = _tiny_linear(seed)
        B, T, D = a.shape
        A, Bc = orc.linear_scan_fwd(a, b)
        for bi in range(B):
            for d in range(D):
                for t in range(T):
                    prod = 1.0
                    for r in range(t + 1):
                        prod *= a[bi, r, d]
                    tot = 0.0
                    for s in range(t + 1):
                        p = 1.0
                        for r in range(s + 1, t + 1):
                            p *= a[bi, r, d]
                        tot += p * b[bi, s, d]
                    assert math.isclose(A[bi, t, d], prod, rel_tol=1e-13, abs_tol=0)
                    assert math.isclose(Bc[bi, t, d], tot, rel_tol=1e-12, abs_tol=1e-13)


def pin_linear_special_cases(orc):
    rng = np.random.default_rng(7)
    b = rng.normal(size=(2, 20, 4))
    A, Bc = orc.linear_scan_fwd(np.ones_like(b), b)
    np.testing.assert_array_equal(A, np.ones_like(b))
    np.testing.assert_allclose(Bc, np.cumsum(b, axis=1), rtol=1e-13, atol=1e-13)
    a = rng.uniform(0.1, 1.5, size=(2, 20, 4))
    A, Bc = orc.linear_scan_fwd(a, np.zeros_like(a))
    np.testing.assert_allclose(A, np.cumprod(a, axis=1), rtol=1e-14, atol=0)
    np.testing.assert_array_equal(Bc, np.zeros_like(a))
    # h_0 folded in: with b_1 = h_0 * a_1 + b_1', h = Bc' + A * h_0
    a, b = _tiny_linear(3)
    h0 = rng.normal(size=(a.shape[0], 1, a.shape[2]))
    A, Bc = orc.linear_scan_fwd(a, b)
    b2 = b.copy()
    b2[:, :1] += a[:, :1] * h0
    _, Bc2 = orc.linear_scan_fwd(a, b2)
    np.testing.assert_allclose(Bc2, Bc + A * h0, rtol=1e-12, atol=1e-12)


def _loss_linear(orc, a, b, gA, gBc):
    A, Bc = orc.linear_scan_fwd(a, b)
    return float(np.sum(gA * A) + np.sum(gBc * Bc))


def pin_linear_adjoint_fd(orc):
    """Central finite differences of L = <gA, A> + <gBc, Bc>, step 1e-6."""
    rng = np.random.default_rng(11)
    a, b = _tiny_linear(5, B=1, T=8, D=2)
    gA, gBc = rng.normal(size=a.shape), rng.normal(size=a.shape)
    A, Bc = orc.linear_scan_fwd(a, b)
    da, db = orc.linear_scan_bwd(a, A, Bc, gA, gBc)
    eps = 1e-6
    for idx in np.ndindex(a.shape):
        for arr, grad in ((a, da), (b, db)):
            old = arr[idx]
            arr[idx] = old + eps
            lp = _loss_linear(orc, a, b, gA, gBc)
            arr[idx] = old - eps
            lm = _loss_linear(orc, a, b, gA, gBc)
            arr[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, grad[idx])


def pin_linear_adjoint_autograd(orc):
    """torch.autograd through the forward recurrence written as a float64 loop."""
    rng = np.random.default_rng(12)
    a, b = _tiny_linear(6, B=2, T=9, D=3)
    gA, gBc = rng.normal(size=a.shape), rng.normal(size=a.shape)
    ta = torch.tensor(a, requires_grad=True)
    tb = torch.tensor(b, requires_grad=True)
    Ap = torch.ones(a.shape[0], a.shape[2], dtype=torch.float64)
    h = torch.zeros_like(Ap)
    As, hs = [], []
    for t in range(a.shape[1]):
        Ap = ta[:, t] * Ap
        h = ta[:, t] * h + tb[:, t]
        As.append(Ap)
        hs.append(h)
    L = (torch.stack(As, 1) * torch.tensor(gA)).sum() + (torch.stack(hs, 1) * torch.tensor(gBc)).sum()
    ga, gb = torch.autograd.grad(L, (ta, tb))
    A, Bc = orc.linear_scan_fwd(a, b)
    da, db = orc.linear_scan_bwd(a, A, Bc, gA, gBc)
    np.testing.assert_allclose(da, ga.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(db, gb.numpy(), rtol=1e-12, atol=1e-12)


def _tiny_log(seed, B=2, T=12, D=3):
    rng = np.random.default_rng(seed)
    lc = -np.log1p(np.exp(rng.normal(size=(B, T, D))))
    lv = rng.normal(size=(B, T + 1, D))
    return lc, lv


def pin_log_vs_linear(orc):
    """log_scan(log a, [log h0, log b]) = Bc + A * h0 of the linear op on a, b."""
    lc, lv = _tiny_log(21)
    h = orc.log_scan_fwd(lc, lv)
    A, Bc = orc.linear_scan_fwd(np.exp(lc), np.exp(lv[:, 1:]))
    h0 = np.exp(lv[:, :1])
    np.testing.assert_allclose(h, Bc + A * h0, rtol=1e-13, atol=0)


def pin_log_closed_form(orc):
    """log h_t = logsumexp_{s=0..t} (lv_s + sum_{r=s+1..t} lc_r), scipy's logsumexp."""
    lc, lv = _tiny_log(22, B=2, T=40, D=2)
    h = orc.log_scan_fwd(lc, lv)
    B, T, D = lc.shape
    for bi in range(B):
        for d in range(D):
            for t in range(1, T + 1):
                terms = [lv[bi, s, d] + sum(lc[bi, r - 1, d] for r in range(s + 1, t + 1))
                         for s in range(t + 1)]
                ref = scipy.special.logsumexp(terms)
                assert math.isclose(math.log(h[bi, t - 1, d]), ref, rel_tol=1e-12, abs_tol=1e-12)


def _rand_mats(rng, shape, k, v):
    A = rng.normal(size=shape + (k, k)) * 0.7
    Bm = rng.normal(size=shape + (k, v))
    return A, Bm


def pin_affine_k1_is_linear(orc):
    a, b = _tiny_linear(31, B=2, T=11, D=3)
    A5 = a[..., None, None]
    B5 = b[..., None, None]
    Abar, Bbar = orc.affine_scan_fwd(A5, B5)
    A, Bc = orc.linear_scan_fwd(a, b)
    np.testing.assert_allclose(Abar[..., 0, 0], A, rtol=1e-14, atol=0)
    np.testing.assert_allclose(Bbar[..., 0, 0], Bc, rtol=1e-13, atol=1e-14)
    rng = np.random.default_rng(32)
    gA, gB = rng.normal(size=a.shape), rng.normal(size=a.shape)
    dA, dB = orc.affine_scan_bwd(A5, Abar, Bbar, gA[..., None, None], gB[..., None, None])
    da, db = orc.linear_scan_bwd(a, A, Bc, gA, gB)
    np.testing.assert_allclose(dA[..., 0, 0], da, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dB[..., 0, 0], db, rtol=1e-12, atol=1e-12)


def pin_affine_diagonal_is_linear(orc):
    """Diagonal A: row i of Bbar is a linear scan with coefficient A[i,i]."""
    rng = np.random.default_rng(33)
    B, T, n, k, v = 1, 10, 2, 3, 2
    diag = rng.uniform(0.3, 1.2, size=(B, T, n, k))
    A = np.zeros((B, T, n, k, k))
    for i in range(k):
        A[..., i, i] = diag[..., i]
    Bm = rng.normal(size=(B, T, n, k, v))
    Abar, Bbar = orc.affine_scan_fwd(A, Bm)
    for ni in range(n):
        for i in range(k):
            a = np.repeat(diag[:, :, ni, i][..., None], v, axis=-1)
            Al, Bl = orc.linear_scan_fwd(a, Bm[:, :, ni, i, :])
            np.testing.assert_allclose(Bbar[:, :, ni, i, :], Bl, rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(Abar[:, :, ni, i, i], Al[..., 0], rtol=1e-14, atol=0)


def pin_affine_running_product(orc):
    """Abar_t = A_t @ ... @ A_1 and Bbar_t = sum_s (A_t ... A_{s+1}) B_s, explicitly."""
    rng = np.random.default_rng(34)
    for (k, v) in ((2, 3), (3, 1), (4, 4)):
        A, Bm = _rand_mats(rng, (2, 7, 2), k, v)
        Abar, Bbar = orc.affine_scan_fwd(A, Bm)
        for bi in range(2):
            for ni in range(2):
                for t in range(7):
                    mats = [A[bi, r, ni] for r in range(t, -1, -1)]  # A_t, ..., A_1
                    P = functools.reduce(np.matmul, mats)
                    np.testing.assert_allclose(Abar[bi, t, ni], P, rtol=1e-12, atol=1e-12)
                    H = np.zeros((k, v))
                    for s in range(t + 1):
                        left = [A[bi, r, ni] for r in range(t, s, -1)]
                        Ls = functools.reduce(np.matmul, left) if left else np.eye(k)
                        H = H + Ls @ Bm[bi, s, ni]
                    np.testing.assert_allclose(Bbar[bi, t, ni], H, rtol=1e-12, atol=1e-12)


def pin_affine_orthogonal_invariant(orc):
    """For A_t = 0.95 Q_t with Q_t orthogonal: Abar_t^T Abar_t = 0.95^(2t) I."""
    from linear_recurrence_scans_gb300.workloads import haar_orthogonal
    for k in (4, 16):
        T = 40
        Q = haar_orthogonal(T * 3, k, seed=5).numpy().reshape(1, T, 3, k, k)
        A = 0.95 * Q
        Abar, _ = orc.affine_scan_fwd(A, np.zeros((1, T, 3, k, 1)))
        for t in range(T):
            G = np.einsum("nij,nil->njl", Abar[0, t], Abar[0, t])
            np.testing.assert_allclose(G, np.broadcast_to(0.95 ** (2 * (t + 1)) * np.eye(k), G.shape),
                                       rtol=0, atol=1e-12)


def _loss_affine(orc, A, Bm, gA, gB):
    Abar, Bbar = orc.affine_scan_fwd(A, Bm)
    return float(np.sum(gA * Abar) + np.sum(gB * Bbar))


def pin_affine_adjoint_fd(orc):
    rng = np.random.default_rng(35)
    for (k, v) in ((2, 3), (3, 2)):
        A, Bm = _rand_mats(rng, (1, 6, 2), k, v)
        gA, gB = rng.normal(size=A.shape), rng.normal(size=Bm.shape)
        Abar, Bbar = orc.affine_scan_fwd(A, Bm)
        dA, dB = orc.affine_scan_bwd(A, Abar, Bbar, gA, gB)
        eps = 1e-6
        for arr, grad in ((A, dA), (Bm, dB)):
            for idx in np.ndindex(arr.shape):
                old = arr[idx]
                arr[idx] = old + eps
                lp = _loss_affine(orc, A, Bm, gA, gB)
                arr[idx] = old - eps
                lm = _loss_affine(orc, A, Bm, gA, gB)
                arr[idx] = old
                fd = (lp - lm) / (2 * eps)
                assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (k, v, idx, fd, grad[idx])


def pin_affine_adjoint_autograd(orc):
    rng = np.random.default_rng(36)
    k, v = 3, 2
    A, Bm = _rand_mats(rng, (2, 8, 2), k, v)
    gA, gB = rng.normal(size=A.shape), rng.normal(size=Bm.shape)
    tA = torch.tensor(A, requires_grad=True)
    tB = torch.tensor(Bm, requires_grad=True)
    P = torch.eye(k, dtype=torch.float64).expand(2, 2, k, k)
    H = torch.zeros(2, 2, k, v, dtype=torch.float64)
    Ps, Hs = [], []
    for t in range(A.shape[1]):
        P = tA[:, t] @ P
        H = tA[:, t] @ H + tB[:, t]
        Ps.append(P)
        Hs.append(H)
    L = (torch.stack(Ps, 1) * torch.tensor(gA)).sum() + (torch.stack(Hs, 1) * torch.tensor(gB)).sum()
    gA_t, gB_t = torch.autograd.grad(L, (tA, tB))
    Abar, Bbar = orc.affine_scan_fwd(A, Bm)
    dA, dB = orc.affine_scan_bwd(A, Abar, Bbar, gA, gB)
    np.testing.assert_allclose(dA, gA_t.numpy(), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(dB, gB_t.numpy(), rtol=1e-11, atol=1e-11)


def pin_golden_log_bwd(orc):
    g = _golden("log_scan_bwd_T2.json")
    lc = np.log(np.array(g["inputs"]["log_coeffs_exp"], dtype=np.float64))
    lv = np.log(np.array(g["inputs"]["log_values_exp"], dtype=np.float64))
    gh = np.array(g["inputs"]["gh"], dtype=np.float64)
    dlc, dlv = orc.log_scan_bwd(lc, lv, gh)
    np.testing.assert_allclose(dlc, np.array(g["expected"]["dlog_coeffs"]), rtol=1e-14)
    np.testing.assert_allclose(dlv, np.array(g["expected"]["dlog_values"]), rtol=1e-14)


def _loss_log(orc, lc, lv, gh):
    return float(np.sum(gh * orc.log_scan_fwd(lc, lv)))


def pin_log_adjoint_fd(orc):
    """Central differences of L = sum(gh * h) in every log input."""
    rng = np.random.default_rng(41)
    lc = -rng.uniform(0.05, 1.5, size=(1, 6, 2))
    lv = rng.normal(scale=0.7, size=(1, 7, 2))
    gh = rng.normal(size=lc.shape)
    dlc, dlv = orc.log_scan_bwd(lc, lv, gh)
    eps = 1e-6
    for arr, grad in ((lc, dlc), (lv, dlv)):
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = _loss_log(orc, lc, lv, gh)
            arr[idx] = old - eps
            lm = _loss_log(orc, lc, lv, gh)
            arr[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, grad[idx])


def pin_log_adjoint_autograd(orc):
    rng = np.random.default_rng(42)
    lc = -rng.uniform(0.05, 2.0, size=(2, 9, 3))
    lv = rng.normal(scale=0.8, size=(2, 10, 3))
    gh = rng.normal(size=lc.shape)
    tlc = torch.tensor(lc, requires_grad=True)
    tlv = torch.tensor(lv, requires_grad=True)
    h = torch.exp(tlv[:, 0])
    hs = []
    for t in range(lc.shape[1]):
        h = torch.exp(tlc[:, t]) * h + torch.exp(tlv[:, t + 1])
        hs.append(h)
    L = (torch.stack(hs, 1) * torch.tensor(gh)).sum()
    g_lc, g_lv = torch.autograd.grad(L, (tlc, tlv))
    dlc, dlv = orc.log_scan_bwd(lc, lv, gh)
    np.testing.assert_allclose(dlc, g_lc.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dlv, g_lv.numpy(), rtol=1e-11, atol=1e-12)


def pin_log_adjoint_vs_linear(orc):
    """The chain rule through the linear op: h = A h0 + Bc with a = exp(lc),
    b = exp(lv[1:]), so dL/dlc = da * a and dL/dlv[1:] = db * b for the
    linear adjoint at gA = gh * h0, gBc = gh, and dL/dlv[0] = h0 sum_t gh_t A_t."""
    rng = np.random.default_rng(43)
    lc = -rng.uniform(0.01, 1.0, size=(2, 30, 4))
    lv = rng.normal(scale=0.5, size=(2, 31, 4))
    gh = rng.normal(size=lc.shape)
    a, b, h0 = np.exp(lc), np.exp(lv[:, 1:]), np.exp(lv[:, :1])
    A, Bc = orc.linear_scan_fwd(a, b)
    da, db = orc.linear_scan_bwd(a, A, Bc, gh * h0, gh)
    dlc, dlv = orc.log_scan_bwd(lc, lv, gh)
    np.testing.assert_allclose(dlc, da * a, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dlv[:, 1:], db * b, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dlv[:, 0], h0[:, 0] * np.sum(gh * A, axis=1), rtol=1e-12, atol=1e-13)


def pin_degenerate_shapes(orc):
    """T = 0 (and empty batch) give empty outputs; T = 1 is a single step."""
    e = np.zeros((2, 0, 3))
    A, Bc = orc.linear_scan_fwd(e, e)
    assert A.shape == (2, 0, 3) and Bc.shape == (2, 0, 3)
    h = orc.log_scan_fwd(e, np.zeros((2, 1, 3)))
    assert h.shape == (2, 0, 3)
    a, b = np.full((1, 1, 2), 0.5), np.array([[[1.0, -2.0]]])
    A, Bc = orc.linear_scan_fwd(a, b)
    np.testing.assert_array_equal(A, a)
    np.testing.assert_array_equal(Bc, b)


# ------------------------------------------- fused minGRU gate + linear scan

def _torch_gate(x1, x2):
    """The minGRU gate written with torch float64 ops (independent of the C)."""
    t1, t2 = torch.as_tensor(x1, dtype=torch.float64), torch.as_tensor(x2, dtype=torch.float64)
    z = torch.sigmoid(t1)
    g = torch.where(t2 >= 0, t2 + 0.5, torch.sigmoid(t2))
    return (1 - z), z * g


def pin_golden_mingru(orc):
    g = _golden("mingru_gate_scan_T2.json")
    gA, gBc = np.array([[[1.0], [0.0]]]), np.array([[[0.0], [1.0]]])
    for case in g["cases"]:
        x1 = np.array(case["x1"]) if "x1" in case else np.log(np.array(case["x1_exp"]))
        x2 = np.array(case["x2"])
        a, b = orc.mingru_gate(x1, x2)
        A, Bc = orc.mingru_scan_fwd(x1, x2)
        dx1, dx2 = orc.mingru_scan_bwd(x1, x2, A, Bc, gA, gBc)
        for name, got in (("a", a), ("b", b), ("A", A), ("Bc", Bc), ("dx1", dx1), ("dx2", dx2)):
            want = np.array(case[name])
            if case["exact"]:
                np.testing.assert_array_equal(got, want, err_msg=f"{case['name']} {name}")
            else:
                np.testing.assert_allclose(got, want, rtol=1e-14, atol=0,
                                           err_msg=f"{case['name']} {name}")


def pin_mingru_gate_vs_torch(orc):
    """The gate against torch's float64 sigmoid, across the range (|x| up to 40,
    where 1 - sigmoid must keep its relative accuracy), and its fixed points."""
    rng = np.random.default_rng(51)
    x1 = np.concatenate([rng.normal(scale=3, size=400), np.linspace(-40, 40, 81)])
    x2 = np.concatenate([rng.normal(scale=3, size=400), np.linspace(-40, 40, 81)])
    a, b = orc.mingru_gate(x1, x2)
    ta = torch.sigmoid(-torch.tensor(x1)).numpy()          # 1 - sigmoid(x1), relatively exact
    _, tb = _torch_gate(x1, x2)
    np.testing.assert_allclose(a, ta, rtol=1e-14, atol=0)
    np.testing.assert_allclose(b, tb.numpy(), rtol=1e-14, atol=0)
    a0, b0 = orc.mingru_gate(np.zeros(3), np.array([0.0, 2.0, -np.inf]))
    np.testing.assert_array_equal(a0, [0.5, 0.5, 0.5])
    np.testing.assert_array_equal(b0, [0.25, 1.25, 0.0])


def pin_mingru_saturated_gate_derivative(orc):
    """For T = 1 with gA = 0, gBc = 1: L = b = z g(x2), so dL/dx1 = z(1-z) g(x2)
    exactly; at |x1| up to 60 (1 - z below double's resolution near 1) the
    oracle must keep its relative accuracy (z(1-z) = e^-|x1| / (1 + e^-|x1|)^2)."""
    x1 = np.array([[[-60.0, -40.0, -5.0, 0.0, 5.0, 40.0, 60.0]]])
    x2 = np.full_like(x1, 1.5)
    A, Bc = orc.mingru_scan_fwd(x1, x2)
    dx1, _ = orc.mingru_scan_bwd(x1, x2, A, Bc, np.zeros_like(x1), np.ones_like(x1))
    e = np.exp(-np.abs(x1))
    np.testing.assert_allclose(dx1, e / (1 + e) ** 2 * 2.0, rtol=1e-13, atol=0)


def pin_mingru_fwd_closed_form(orc):
    """A and Bc of the fused op by brute-force products and sums of torch's gate."""
    rng = np.random.default_rng(52)
    x1, x2 = rng.normal(size=(2, 9, 3)), rng.normal(size=(2, 9, 3))
    a, b = (t.numpy() for t in _torch_gate(x1, x2))
    A, Bc = orc.mingru_scan_fwd(x1, x2)
    Bn, T, D = x1.shape
    for bi in range(Bn):
        for d in range(D):
            for t in range(T):
                prod = float(np.prod(a[bi, :t + 1, d]))
                tot = sum(float(np.prod(a[bi, s + 1:t + 1, d])) * b[bi, s, d] for s in range(t + 1))
                assert math.isclose(A[bi, t, d], prod, rel_tol=1e-13, abs_tol=0)
                assert math.isclose(Bc[bi, t, d], tot, rel_tol=1e-12, abs_tol=1e-14)


def _loss_mingru(orc, x1, x2, gA, gBc):
    A, Bc = orc.mingru_scan_fwd(x1, x2)
    return float(np.sum(gA * A) + np.sum(gBc * Bc))


def pin_mingru_adjoint_fd(orc):
    """Central differences of L in every x1, x2 (x2 kept off g's branch point)."""
    rng = np.random.default_rng(53)
    x1 = rng.normal(size=(1, 7, 2))
    x2 = rng.normal(size=(1, 7, 2))
    x2 = np.where(np.abs(x2) < 0.05, 0.3, x2)
    gA, gBc = rng.normal(size=x1.shape), rng.normal(size=x1.shape)
    A, Bc = orc.mingru_scan_fwd(x1, x2)
    dx1, dx2 = orc.mingru_scan_bwd(x1, x2, A, Bc, gA, gBc)
    eps = 1e-6
    for arr, grad in ((x1, dx1), (x2, dx2)):
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = _loss_mingru(orc, x1, x2, gA, gBc)
            arr[idx] = old - eps
            lm = _loss_mingru(orc, x1, x2, gA, gBc)
            arr[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, grad[idx])


def pin_mingru_adjoint_autograd(orc):
    """torch.autograd through the gate and a float64 recurrence loop."""
    rng = np.random.default_rng(54)
    x1, x2 = rng.normal(size=(2, 8, 3)), rng.normal(size=(2, 8, 3))
    x2[0, 3, 1] = 0.0                 # g's branch point: its derivative is that of x + 0.5
    gA, gBc = rng.normal(size=x1.shape), rng.normal(size=x1.shape)
    t1 = torch.tensor(x1, requires_grad=True)
    t2 = torch.tensor(x2, requires_grad=True)
    a, b = _torch_gate(t1, t2)
    Ap = torch.ones(2, 3, dtype=torch.float64)
    h = torch.zeros_like(Ap)
    As, hs = [], []
    for t in range(8):
        Ap = a[:, t] * Ap
        h = a[:, t] * h + b[:, t]
        As.append(Ap)
        hs.append(h)
    L = (torch.stack(As, 1) * torch.tensor(gA)).sum() + (torch.stack(hs, 1) * torch.tensor(gBc)).sum()
    g1, g2 = torch.autograd.grad(L, (t1, t2))
    A, Bc = orc.mingru_scan_fwd(x1, x2)
    dx1, dx2 = orc.mingru_scan_bwd(x1, x2, A, Bc, gA, gBc)
    np.testing.assert_allclose(dx1, g1.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dx2, g2.numpy(), rtol=1e-12, atol=1e-13)


# ------------------------------------------ start states, varlen batches

def pin_golden_varlen_h0(orc):
    g = _golden("linear_scan_varlen_h0.json")
    a, b, h0 = np.array(g["a"]), np.array(g["b"]), np.array(g["h0"])
    A, H = orc.linear_scan_varlen_fwd(a, b, g["cu_seqlens"], h0)
    np.testing.assert_array_equal(A, np.array(g["A"]))
    np.testing.assert_array_equal(H, np.array(g["H"]))
    da, db, dh0 = orc.linear_scan_varlen_bwd(a, g["cu_seqlens"], A, H, np.array(g["gA"]),
                                             np.array(g["gH"]), h0)
    np.testing.assert_array_equal(da, np.array(g["da"]))
    np.testing.assert_array_equal(db, np.array(g["db"]))
    np.testing.assert_array_equal(dh0, np.array(g["dh0"]))


def _packed(rng, lens, D):
    cu = np.concatenate([[0], np.cumsum(lens)])
    a = rng.uniform(0.2, 1.3, (cu[-1], D)) * rng.choice([-1, 1], (cu[-1], D))
    b = rng.normal(size=(cu[-1], D))
    return a, b, cu


def pin_varlen_is_independent_scans(orc):
    """Each packed sequence is the plain scan of its own rows: without h0 the
    linear op's (A, Bc) and adjoint; with h0, H = Bc + A h0 (the start state
    carried by the running product) and A unchanged."""
    rng = np.random.default_rng(61)
    lens = [5, 0, 1, 9, 3]
    a, b, cu = _packed(rng, lens, 3)
    h0 = rng.normal(size=(len(lens), 3))
    gA, gH = rng.normal(size=a.shape), rng.normal(size=a.shape)
    A0, H0 = orc.linear_scan_varlen_fwd(a, b, cu)
    A1, H1 = orc.linear_scan_varlen_fwd(a, b, cu, h0)
    da0, db0, dh = orc.linear_scan_varlen_bwd(a, cu, A0, H0, gA, gH)
    assert dh is None
    for s in range(len(lens)):
        r0, r1 = cu[s], cu[s + 1]
        if r1 == r0:
            continue
        A, Bc = orc.linear_scan_fwd(a[None, r0:r1], b[None, r0:r1])
        np.testing.assert_array_equal(A0[r0:r1], A[0])
        np.testing.assert_array_equal(H0[r0:r1], Bc[0])
        np.testing.assert_array_equal(A1[r0:r1], A[0])
        np.testing.assert_allclose(H1[r0:r1], Bc[0] + A[0] * h0[s], rtol=1e-12, atol=1e-12)
        da, db = orc.linear_scan_bwd(a[None, r0:r1], A, Bc, gA[None, r0:r1], gH[None, r0:r1])
        np.testing.assert_array_equal(da0[r0:r1], da[0])
        np.testing.assert_array_equal(db0[r0:r1], db[0])


def pin_h0_batch_is_varlen(orc):
    """The (B,T,D) form with h0 (B,D) against the identity H = Bc + A h0 of the
    plain op (a start state folded into the first value, b_1 + a_1 h0)."""
    rng = np.random.default_rng(62)
    a, b = _tiny_linear(63, B=3, T=7, D=2)
    h0 = rng.normal(size=(3, 2))
    A, H = orc.linear_scan_h0_fwd(a, b, h0)
    b2 = b.copy()
    b2[:, 0] += a[:, 0] * h0
    A2, Bc2 = orc.linear_scan_fwd(a, b2)
    np.testing.assert_array_equal(A, A2)
    np.testing.assert_allclose(H, Bc2, rtol=1e-13, atol=1e-13)


def _loss_varlen(orc, a, b, cu, h0, gA, gH):
    A, H = orc.linear_scan_varlen_fwd(a, b, cu, h0)
    return float(np.sum(gA * A) + np.sum(gH * H))


def pin_varlen_adjoint_fd(orc):
    rng = np.random.default_rng(64)
    a, b, cu = _packed(rng, [4, 0, 3, 1], 2)
    h0 = rng.normal(size=(4, 2))
    gA, gH = rng.normal(size=a.shape), rng.normal(size=a.shape)
    A, H = orc.linear_scan_varlen_fwd(a, b, cu, h0)
    da, db, dh0 = orc.linear_scan_varlen_bwd(a, cu, A, H, gA, gH, h0)
    eps = 1e-6
    for arr, grad in ((a, da), (b, db), (h0, dh0)):
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = _loss_varlen(orc, a, b, cu, h0, gA, gH)
            arr[idx] = old - eps
            lm = _loss_varlen(orc, a, b, cu, h0, gA, gH)
            arr[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, grad[idx])


def pin_golden_affine_h0(orc):
    g = _golden("affine_scan_h0_k2.json")
    A, Bm, H0 = np.array(g["A"]), np.array(g["Bm"]), np.array(g["H0"])
    Abar, Bbar = orc.affine_scan_h0_fwd(A, Bm, H0)
    np.testing.assert_array_equal(Abar, np.array(g["Abar"]))
    np.testing.assert_array_equal(Bbar, np.array(g["Bbar"]))
    dA, dB, dH0 = orc.affine_scan_h0_bwd(A, H0, Abar, Bbar, np.array(g["gAbar"]),
                                         np.array(g["gBbar"]))
    np.testing.assert_array_equal(dA, np.array(g["dA"]))
    np.testing.assert_array_equal(dB, np.array(g["dB"]))
    np.testing.assert_array_equal(dH0, np.array(g["dH0"]))


def pin_affine_h0_identity(orc):
    """Bbar(H0) = Bbar(0) + Abar H0 (numpy matmul); Abar does not depend on H0;
    H0 = 0 gives the plain op and its adjoint."""
    rng = np.random.default_rng(65)
    for (k, v) in ((2, 3), (4, 1), (3, 3)):
        A, Bm = _rand_mats(rng, (2, 6, 3), k, v)
        H0 = rng.normal(size=(2, 3, k, v))
        Abar, Bbar = orc.affine_scan_h0_fwd(A, Bm, H0)
        Abar0, Bbar0 = orc.affine_scan_fwd(A, Bm)
        np.testing.assert_array_equal(Abar, Abar0)
        np.testing.assert_allclose(Bbar, Bbar0 + Abar @ H0[:, None], rtol=1e-12, atol=1e-12)
        gA, gB = rng.normal(size=A.shape), rng.normal(size=Bm.shape)
        Z = np.zeros_like(H0)
        Ab, Bb = orc.affine_scan_h0_fwd(A, Bm, Z)
        dA, dB, _ = orc.affine_scan_h0_bwd(A, Z, Ab, Bb, gA, gB)
        dA0, dB0 = orc.affine_scan_bwd(A, Abar0, Bbar0, gA, gB)
        np.testing.assert_array_equal(dA, dA0)
        np.testing.assert_array_equal(dB, dB0)


def _loss_affine_h0(orc, A, Bm, H0, gA, gB):
    Abar, Bbar = orc.affine_scan_h0_fwd(A, Bm, H0)
    return float(np.sum(gA * Abar) + np.sum(gB * Bbar))


def pin_affine_h0_adjoint_fd(orc):
    rng = np.random.default_rng(66)
    k, v = 2, 3
    A, Bm = _rand_mats(rng, (1, 5, 2), k, v)
    H0 = rng.normal(size=(1, 2, k, v))
    gA, gB = rng.normal(size=A.shape), rng.normal(size=Bm.shape)
    Abar, Bbar = orc.affine_scan_h0_fwd(A, Bm, H0)
    dA, dB, dH0 = orc.affine_scan_h0_bwd(A, H0, Abar, Bbar, gA, gB)
    eps = 1e-6
    for arr, grad in ((A, dA), (Bm, dB), (H0, dH0)):
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = _loss_affine_h0(orc, A, Bm, H0, gA, gB)
            arr[idx] = old - eps
            lm = _loss_affine_h0(orc, A, Bm, H0, gA, gB)
            arr[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, grad[idx])


def pin_new_degenerate_shapes(orc):
    """Empty sequences and empty batches; T = 0 with H0 gives dH0 = 0."""
    e = np.zeros((0, 3))
    A, H = orc.linear_scan_varlen_fwd(e, e, [0, 0, 0], np.ones((2, 3)))
    assert A.shape == (0, 3)
    _, _, dh0 = orc.linear_scan_varlen_bwd(e, [0, 0, 0], e, e, e, e, np.ones((2, 3)))
    np.testing.assert_array_equal(dh0, np.zeros((2, 3)))
    A5 = np.zeros((1, 0, 2, 3, 3))
    B5 = np.zeros((1, 0, 2, 3, 1))
    H0 = np.ones((1, 2, 3, 1))
    Ab, Bb = orc.affine_scan_h0_fwd(A5, B5, H0)
    _, _, dH0 = orc.affine_scan_h0_bwd(A5, H0, Ab, Bb, A5, B5)
    np.testing.assert_array_equal(dH0, np.zeros_like(H0))


# ----------------------------------------------- angle-fused scan (reading)

def _angle_inputs(rng, B, T, n, R, k, sgn_pm=True):
    theta = rng.uniform(-np.pi, np.pi, size=(B, T, n, R, k // 2))
    scale = np.tanh(rng.normal(size=(B, T, n)))
    gamma = np.exp(-rng.uniform(0.0, 0.3, size=(B, T, n)))
    b = rng.normal(size=(B, T, n, k))
    h0 = rng.normal(size=(B, n, k))
    perm = np.stack([rng.permutation(k) for _ in range(R)]).astype(np.int32)
    sgn = rng.choice([-1.0, 1.0], size=(R, k)) if sgn_pm else rng.uniform(0.5, 1.5, size=(R, k))
    return theta, scale, gamma, b, h0, perm, sgn


def _angle_dense(theta, perm, sgn, deriv=None):
    """Q_t of every step as an explicit k x k product of Givens matrices
    (numpy); with deriv = (r, i), the derivative of Q_t in theta_{t,r,i}."""
    B, T, n, R, half = theta.shape
    k = 2 * half
    Q = np.zeros((B, T, n, k, k))
    for idx in np.ndindex(B, T, n):
        M = np.eye(k)
        for r in range(R):
            G = np.eye(k)
            for i in range(half):
                p, q = perm[r][2 * i], perm[r][2 * i + 1]
                c, s_ = np.cos(theta[idx + (r, i)]), np.sin(theta[idx + (r, i)])
                if deriv == (r, i):
                    G[p, p], G[p, q], G[q, p], G[q, q] = -s_, -c, c, -s_
                else:
                    G[p, p], G[p, q], G[q, p], G[q, q] = c, -s_, s_, c
            if deriv is not None and deriv[0] == r:
                for i in range(half):                   # the other pairs do not move
                    if i != deriv[1]:
                        p, q = perm[r][2 * i], perm[r][2 * i + 1]
                        G[p, p] = G[p, q] = G[q, p] = G[q, q] = 0.0
                for j in range(k):
                    if j not in (perm[r][2 * deriv[1]], perm[r][2 * deriv[1] + 1]):
                        G[j, j] = 0.0
            M = np.diag(sgn[r]) @ G @ M
        Q[idx] = M
    return Q


def pin_golden_angle(orc):
    g = _golden("angle_scan_k2.json")
    a = {k_: np.array(g[k_]) for k_ in ("theta", "scale", "gamma", "b", "h0", "sgn", "grad_out")}
    h = orc.angle_scan_fwd(a["theta"], a["scale"], a["gamma"], a["b"], a["h0"], g["perm"], a["sgn"])
    np.testing.assert_allclose(h, np.array(g["h"]), rtol=1e-14, atol=1e-15)
    r = orc.angle_scan_bwd(a["theta"], a["scale"], a["gamma"], a["h0"], np.array(g["h"]),
                           a["grad_out"], g["perm"], a["sgn"])
    for name, got in zip(("dtheta", "dscale", "dgamma", "db", "dh0"), r):
        np.testing.assert_allclose(got, np.array(g[name]), rtol=1e-14, atol=1e-15, err_msg=name)


def pin_angle_vs_dense_affine(orc):
    """The scan equals the affine scan (pinned above) on the explicit dense
    transitions A_t = s g Q_t with a vector state, and its gradients are the
    affine adjoint's carried through A_t by matrix calculus:
    dscale = g <dA, Q>, dgamma = s <dA, Q>, dtheta = s g <dA, dQ/dtheta>."""
    rng = np.random.default_rng(71)
    B, T, n, R, k = 2, 6, 2, 3, 4
    th, sc, ga, b, h0, perm, sgn = _angle_inputs(rng, B, T, n, R, k, sgn_pm=False)
    Q = _angle_dense(th, perm, sgn)
    A = (sc * ga)[..., None, None] * Q
    h = orc.angle_scan_fwd(th, sc, ga, b, h0, perm, sgn)
    _, Hb = orc.affine_scan_h0_fwd(A, b[..., None], h0[..., None])
    np.testing.assert_allclose(h, Hb[..., 0], rtol=1e-12, atol=1e-12)
    go = rng.normal(size=h.shape)
    Abar, _ = orc.affine_scan_h0_fwd(A, b[..., None], h0[..., None])
    dA, dB, dH0 = orc.affine_scan_h0_bwd(A, h0[..., None], Abar, h[..., None],
                                         np.zeros_like(Abar), go[..., None])
    dth, dsc, dga, db, dh0 = orc.angle_scan_bwd(th, sc, ga, h0, h, go, perm, sgn)
    np.testing.assert_allclose(db, dB[..., 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dh0, dH0[..., 0], rtol=1e-12, atol=1e-12)
    inner = np.sum(dA * Q, axis=(-2, -1))
    np.testing.assert_allclose(dsc, ga * inner, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dga, sc * inner, rtol=1e-11, atol=1e-12)
    for r in range(R):
        for i in range(k // 2):
            dQ = _angle_dense(th, perm, sgn, deriv=(r, i))
            want = sc * ga * np.sum(dA * dQ, axis=(-2, -1))
            np.testing.assert_allclose(dth[..., r, i], want, rtol=1e-10, atol=1e-11)


def pin_angle_special_cases(orc):
    """theta = 0, sgn = 1: Q = I and every coordinate is the linear scan with
    a = s g from h0; scale and gamma are ignored (and their gradients zero)
    without has_scale / has_decay; b = 0, s = g = 1, sgn = +-1 keep |h_t| = |h0|."""
    rng = np.random.default_rng(72)
    B, T, n, R, k = 2, 7, 3, 2, 4
    th, sc, ga, b, h0, perm, sgn = _angle_inputs(rng, B, T, n, R, k)
    h = orc.angle_scan_fwd(np.zeros_like(th), sc, ga, b, h0, perm, np.ones_like(sgn))
    a = np.repeat((sc * ga)[..., None], k, axis=-1)
    _, H = orc.linear_scan_h0_fwd(a.reshape(B, T, n * k), b.reshape(B, T, n * k),
                                  h0.reshape(B, n * k))
    np.testing.assert_allclose(h, H.reshape(h.shape), rtol=1e-12, atol=1e-12)
    h1 = orc.angle_scan_fwd(th, sc, ga, b, h0, perm, sgn, has_scale=0, has_decay=0)
    h2 = orc.angle_scan_fwd(th, sc * 3 + 1, ga * 0.1, b, h0, perm, sgn, has_scale=0, has_decay=0)
    np.testing.assert_array_equal(h1, h2)
    go = rng.normal(size=h1.shape)
    _, dsc, dga, _, _ = orc.angle_scan_bwd(th, sc, ga, h0, h1, go, perm, sgn, 0, 0)
    assert not dsc.any() and not dga.any()
    hn = orc.angle_scan_fwd(th, np.ones_like(sc), np.ones_like(ga), np.zeros_like(b), h0, perm, sgn)
    np.testing.assert_allclose(np.linalg.norm(hn, axis=-1),
                               np.broadcast_to(np.linalg.norm(h0, axis=-1)[:, None], hn.shape[:-1]),
                               rtol=1e-12)


def _loss_angle(orc, th, sc, ga, b, h0, perm, sgn, go):
    return float(np.sum(go * orc.angle_scan_fwd(th, sc, ga, b, h0, perm, sgn)))


def pin_angle_adjoint_fd(orc):
    rng = np.random.default_rng(73)
    th, sc, ga, b, h0, perm, sgn = _angle_inputs(rng, 1, 5, 2, 2, 4, sgn_pm=False)
    h = orc.angle_scan_fwd(th, sc, ga, b, h0, perm, sgn)
    go = rng.normal(size=h.shape)
    grads = orc.angle_scan_bwd(th, sc, ga, h0, h, go, perm, sgn)
    eps = 1e-6
    for arr, grad in zip((th, sc, ga, b, h0), grads):
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = _loss_angle(orc, th, sc, ga, b, h0, perm, sgn, go)
            arr[idx] = old - eps
            lm = _loss_angle(orc, th, sc, ga, b, h0, perm, sgn, go)
            arr[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, grad[idx])


def pin_angle_adjoint_autograd(orc):
    """torch.autograd through the reading written as a float64 torch loop."""
    rng = np.random.default_rng(74)
    B, T, n, R, k = 2, 6, 2, 3, 8
    th, sc, ga, b, h0, perm, sgn = _angle_inputs(rng, B, T, n, R, k)
    t = {nm: torch.tensor(x, requires_grad=True) for nm, x in
         (("th", th), ("sc", sc), ("ga", ga), ("b", b), ("h0", h0))}
    x = t["h0"]
    hs = []
    for ti in range(T):
        for r in range(R):
            cols = list(x.unbind(-1))
            for i in range(k // 2):
                p, q = int(perm[r][2 * i]), int(perm[r][2 * i + 1])
                c, s_ = torch.cos(t["th"][:, ti, :, r, i]), torch.sin(t["th"][:, ti, :, r, i])
                cols[p], cols[q] = c * cols[p] - s_ * cols[q], s_ * cols[p] + c * cols[q]
            x = torch.stack(cols, -1) * torch.tensor(sgn[r])
        x = (t["sc"][:, ti] * t["ga"][:, ti])[..., None] * x + t["b"][:, ti]
        hs.append(x)
    h = torch.stack(hs, 1)
    go = rng.normal(size=h.shape)
    L = (h * torch.tensor(go)).sum()
    want = torch.autograd.grad(L, [t[nm] for nm in ("th", "sc", "ga", "b", "h0")])
    hh = orc.angle_scan_fwd(th, sc, ga, b, h0, perm, sgn)
    np.testing.assert_allclose(hh, h.detach().numpy(), rtol=1e-12, atol=1e-12)
    got = orc.angle_scan_bwd(th, sc, ga, h0, hh, go, perm, sgn)
    for nm, g_, w in zip(("th", "sc", "ga", "b", "h0"), got, want):
        np.testing.assert_allclose(g_, w.numpy(), rtol=1e-11, atol=1e-11, err_msg=nm)


PINS = [
    pin_golden_linear, pin_golden_log, pin_golden_affine,
    pin_linear_closed_form, pin_linear_special_cases,
    pin_linear_adjoint_fd, pin_linear_adjoint_autograd,
    pin_log_vs_linear, pin_log_closed_form,
    pin_golden_log_bwd, pin_log_adjoint_fd, pin_log_adjoint_autograd, pin_log_adjoint_vs_linear,
    pin_affine_k1_is_linear, pin_affine_diagonal_is_linear,
    pin_affine_running_product, pin_affine_orthogonal_invariant,
    pin_affine_adjoint_fd, pin_affine_adjoint_autograd,
    pin_degenerate_shapes,
    pin_golden_mingru, pin_mingru_gate_vs_torch, pin_mingru_fwd_closed_form,
    pin_mingru_saturated_gate_derivative,
    pin_mingru_adjoint_fd, pin_mingru_adjoint_autograd,
    pin_golden_varlen_h0, pin_varlen_is_independent_scans, pin_h0_batch_is_varlen,
    pin_varlen_adjoint_fd, pin_golden_affine_h0, pin_affine_h0_identity,
    pin_affine_h0_adjoint_fd, pin_new_degenerate_shapes,
    pin_golden_angle, pin_angle_vs_dense_affine, pin_angle_special_cases,
    pin_angle_adjoint_fd, pin_angle_adjoint_autograd,
]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle._oracle())


# Plausible mistakes, planted in copies of the oracle's C source (in every
# function where the line occurs).  Each must make at least one pin fail.
MUTANTS = {
    "linear_fwd_dropped_coefficient": ("h[d] = at * h[d] + b[row + d];", "h[d] = h[d] + b[row + d];"),
    "linear_fwd_exclusive_product": ("A[row + d] = Ap[d];", "A[row + d] = Ap[d] / at;"),
    "linear_bwd_coefficient_index": ("a[row + D + d] : 0.0", "a[row + d] : 0.0"),
    "linear_bwd_dropped_term": ("da[row + d] = mu[d] * A_prev + lam[d] * Bc_prev;",
                                "da[row + d] = mu[d] * A_prev;"),
    "linear_bwd_sign": ("mu[d] = gA[row + d] + a_next * mu[d];", "mu[d] = gA[row + d] - a_next * mu[d];"),
    "linear_bwd_halo_index": ("const double A_prev = (t > 0) ? A[row - D + d] : 1.0;",
                              "const double A_prev = (t > 0) ? A[row + d] : 1.0;"),
    "log_value_slot": ("exp(log_values[vrow + d])", "exp(log_values[vrow - D + d])"),
    "log_dropped_h0": ("h[d] = exp(log_values[v0 + d]);", "h[d] = 0.0;"),
    "log_bwd_coefficient_index": ("const double a_next = t < T ? exp(log_coeffs[crow + D]) : 0.0;",
                                  "const double a_next = t < T ? exp(log_coeffs[crow]) : 0.0;"),
    "log_bwd_halo_index": ("dlog_coeffs[crow] = mu * exp(log_coeffs[crow]) * h[t - 1];",
                           "dlog_coeffs[crow] = mu * exp(log_coeffs[crow]) * h[t];"),
    "log_bwd_dropped_slot0": ("dlog_values[v0] = T >= 1 ? exp(log_coeffs[(bi * T) * D + d]) * mu * h[0] : 0.0;",
                              "dlog_values[v0] = 0.0;"),
    "linear_fwd_product_from_zero": ("            Ap[d] = 1.0;\n", "            Ap[d] = 0.0;\n"),
    "log_fwd_coefficient_sign": ("h[d] = exp(log_coeffs[crow + d]) * h[d] + exp(log_values[vrow + d]);",
                                 "h[d] = exp(-log_coeffs[crow + d]) * h[d] + exp(log_values[vrow + d]);"),
    "affine_bwd_coefficient_index": ("const double *Anext = A + (s + n) * kk;",
                                     "const double *Anext = A + s * kk;"),
    "affine_bwd_halo_index": ("const double *Aprev = (t > 0) ? Abar + (s - n) * kk : eye;",
                              "const double *Aprev = (t > 0) ? Abar + s * kk : eye;"),
    "affine_fwd_order": ("mat_mul(At, P, tmp, k, k, k);", "mat_mul(P, At, tmp, k, k, k);"),
    "affine_fwd_dropped_B": ("H[e] = tmp[e] + Bm[s * kv + e];", "H[e] = tmp[e];"),
    "affine_bwd_untransposed": ("mat_tmul(Anext, M, tmp, k, k, k);", "mat_mul(Anext, M, tmp, k, k, k);"),
    "affine_bwd_dropped_term": ("mat_mul_tadd(L, Bprev, dAt, k, v, k);", ""),
    "matmul_transposed_operand": ("s += X[i * m + l] * Y[l * c + j];", "s += X[l * m + i] * Y[l * c + j];"),
    "gate_coefficient_sign": ("a[i] = orc_sigmoid(-x1[i]);", "a[i] = orc_sigmoid(x1[i]);"),
    "gate_g_branch": ("return x >= 0.0 ? x + 0.5 : orc_sigmoid(x);",
                      "return x >= 0.0 ? x + 0.5 : orc_sigmoid(-x);"),
    "gate_g_grad_at_positive": ("if (x >= 0.0) return 1.0;", "if (x >= 0.0) return 0.5;"),
    "gate_bwd_dx1_sign": ("dx1[i] = (db[i] * orc_g(x2[i]) - da[i]) * z * zc;",
                          "dx1[i] = (db[i] * orc_g(x2[i]) + da[i]) * z * zc;"),
    "gate_bwd_dx1_dropped_zc": ("dx1[i] = (db[i] * orc_g(x2[i]) - da[i]) * z * zc;",
                                "dx1[i] = (db[i] * orc_g(x2[i]) - da[i]) * z;"),
    "gate_bwd_dx2_dropped_z": ("dx2[i] = db[i] * z * orc_g_grad(x2[i]);",
                               "dx2[i] = db[i] * orc_g_grad(x2[i]);"),
    "varlen_dropped_h0": ("double Ap = 1.0, h = h0 ? h0[s * D + d] : 0.0;", "double Ap = 1.0, h = 0.0;"),
    "varlen_bwd_start_state": ("(h0 ? h0[s * D + d] : 0.0)", "0.0"),
    "varlen_bwd_crosses_sequences": ("const double A_prev = (r > r0) ? A[(r - 1) * D + d] : 1.0;",
                                     "const double A_prev = (r > 0) ? A[(r - 1) * D + d] : 1.0;"),
    "varlen_dh0_index": ("a[r0 * D + d] * lam", "a[(r1 - 1) * D + d] * lam"),
    "affine_h0_dropped": ("memcpy(Hs, H0 + (bi * n + ni) * kv, (size_t)kv * sizeof(double));",
                          "memset(Hs, 0, (size_t)kv * sizeof(double));"),
    "affine_h0_bwd_start_state": ("const double *Bprev = (t > 0) ? Bbar + (s - n) * kv : h0;",
                                  "const double *Bprev = (t > 0) ? Bbar + (s - n) * kv : Bbar + s * kv;"),
    "affine_dh0_untransposed": ("mat_tmul(A + ((bi * T) * n + ni) * kk, L, dh, k, k, v);",
                                "mat_mul(A + ((bi * T) * n + ni) * kk, L, dh, k, k, v);"),
    "angle_rotation_sign": ("x[p] = c * xp - s * xq;", "x[p] = c * xp + s * xq;"),
    "angle_dropped_signs": ("            x[j] *= sgn[r * k + j];\n", "            x[j] *= 1.0;\n"),
    "angle_bwd_dtheta_sign": ("u[p] * (-sn * x[p] - c * x[q])", "u[p] * (sn * x[p] - c * x[q])"),
    "angle_bwd_untransposed": ("u[p] = c * up + sn * uq;", "u[p] = c * up - sn * uq;"),
    "angle_bwd_dscale_without_gamma": ("dscale[s] = has_scale ? ga * dot : 0.0;",
                                       "dscale[s] = has_scale ? dot : 0.0;"),
    "angle_bwd_halo_index": ("const double *hp = t > 0 ? out + (s - n) * k",
                             "const double *hp = t > 0 ? out + s * k"),
    "angle_decay_flag_ignored": ("(has_decay ? gamma[s] : 1.0)", "(gamma[s])"),
}


def test_planted_mistakes_are_caught():
    src = open(oracle._SRC).read()
    tmp = tempfile.mkdtemp(prefix="orc_mut_")
    try:
        for name, (old, new) in MUTANTS.items():
            assert src.count(old) >= 1, name   # planted wherever the line occurs
            path = os.path.join(tmp, f"{name}.c")
            with open(path, "w") as f:
                f.write(src.replace(old, new))
            orc = oracle.Oracle(oracle.build(force=True, src=path, out=path[:-2] + ".so"))
            caught = []
            for pin in PINS:
                try:
                    pin(orc)
                except AssertionError:
                    caught.append(pin.__name__)
            assert caught, f"planted mistake {name} passed every pin"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
