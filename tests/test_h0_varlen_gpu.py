"""GPU parity of the linear scan from start states (mg_linear_scan_h0_fwd/bwd)
and over packed variable-length batches (mg_linear_scan_varlen_fwd/bwd)
against the float64 oracle, through the C ABI (via the Python binding).
Outputs start as NaN so an unwritten element fails."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from linear_recurrence_scans_gb300 import workloads as wl
from parity import TOL_BF16, TOL_F32, scaled_error

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _nan(shape):
    return torch.full(tuple(shape), float("nan"), device=DEV)


def _np(x):
    return x.detach().to("cpu", torch.float64).numpy()


def _h0_case(mg, a, b, h0, gA, gH, tol):
    import oracle
    ad, bd, hd = a.to(DEV), b.to(DEV), h0.to(DEV)
    A, H = mg.linear_scan_h0_fwd(ad, bd, hd, out=(_nan(a.shape), _nan(a.shape)))
    rA, rH = oracle.linear_scan_h0_fwd(a, b, h0)
    SA, SH = oracle.linear_scan_h0_fwd(np.abs(_np(a)), np.abs(_np(b)), np.abs(_np(h0)))
    errs = {"A": scaled_error(_np(A), rA, SA), "H": scaled_error(_np(H), rH, SH)}
    assert max(errs.values()) <= tol, errs
    A32, H32 = torch.from_numpy(rA).float(), torch.from_numpy(rH).float()
    da, db, dh0 = mg.linear_scan_h0_bwd(ad, hd, A32.to(DEV), H32.to(DEV), gA.to(DEV), gH.to(DEV),
                                        out=(_nan(a.shape), _nan(a.shape), _nan(h0.shape)))
    r = oracle.linear_scan_h0_bwd(a, h0, A32, H32, gA, gH)
    S = oracle.linear_scan_h0_bwd(*(np.abs(_np(x)) for x in (a, h0, A32, H32, gA, gH)))
    eb = {k: scaled_error(_np(g), rr, ss) for k, g, rr, ss in zip(("da", "db", "dh0"),
                                                                 (da, db, dh0), r, S)}
    assert max(eb.values()) <= tol, eb
    mg.workspace_status()
    return {**errs, **eb}


@pytest.mark.parametrize("shape", [(1, 1, 4), (3, 517, 300), (2, 1000, 37), (1, 4099, 8),
                                   (8, 4096, 1024)])
def test_h0_fp32(cuda_lib, shape):
    a, b, gA, gH = wl.mingru_linear(*shape, seed=41)
    h0 = torch.randn(shape[0], shape[2], generator=torch.Generator().manual_seed(42))
    _h0_case(cuda_lib, a, b, h0, gA, gH, TOL_F32)


@pytest.mark.parametrize("shape", [(2, 300, 256), (1, 50, 13)])
def test_h0_bf16(cuda_lib, shape):
    a, b, gA, gH = wl.mingru_linear(*shape, seed=43, in_dtype=torch.bfloat16)
    h0 = torch.randn(shape[0], shape[2], generator=torch.Generator().manual_seed(44))
    _h0_case(cuda_lib, a, b, h0, gA, gH, TOL_F32)


def test_h0_zero_equals_plain_op(cuda_lib):
    """h0 = 0 gives bitwise the plain op (same tiles, same combine order)."""
    mg = cuda_lib
    a, b, gA, gH = wl.mingru_linear(2, 700, 256, seed=45, device=DEV)
    z = torch.zeros(2, 256, device=DEV)
    A, H = mg.linear_scan_h0_fwd(a, b, z)
    A0, Bc0 = mg.linear_scan_fwd(a, b)
    assert torch.equal(A, A0) and torch.equal(H, Bc0)
    da, db, dh0 = mg.linear_scan_h0_bwd(a, z, A, H, gA, gH)
    da0, db0 = mg.linear_scan_bwd(a, A, H, gA, gH)
    assert torch.equal(da, da0) and torch.equal(db, db0)


def _lens(rng, n, lo, hi, empty_every=0):
    lens = rng.integers(lo, hi, size=n)
    if empty_every:
        lens[::empty_every] = 0
    return lens


def _varlen_case(mg, a, b, cu, h0, gA, gH, tol):
    import oracle
    ad, bd = a.to(DEV), b.to(DEV)
    cut = torch.as_tensor(cu, dtype=torch.int64)
    hd = None if h0 is None else h0.to(DEV)
    A, H = mg.linear_scan_varlen_fwd(ad, bd, cut, hd, out=(_nan(a.shape), _nan(a.shape)))
    rA, rH = oracle.linear_scan_varlen_fwd(a, b, cu, h0)
    SA, SH = oracle.linear_scan_varlen_fwd(np.abs(_np(a)), np.abs(_np(b)), cu,
                                           None if h0 is None else np.abs(_np(h0)))
    errs = {"A": scaled_error(_np(A), rA, SA), "H": scaled_error(_np(H), rH, SH)}
    assert max(errs.values()) <= tol, errs
    A32, H32 = torch.from_numpy(rA).float(), torch.from_numpy(rH).float()
    nseq = len(cu) - 1
    outs = (_nan(a.shape), _nan(a.shape), None if h0 is None else _nan((nseq, a.shape[1])))
    da, db, dh0 = mg.linear_scan_varlen_bwd(ad, cut, A32.to(DEV), H32.to(DEV), gA.to(DEV),
                                            gH.to(DEV), hd, out=outs)
    r = oracle.linear_scan_varlen_bwd(a, cu, A32, H32, gA, gH, h0)
    S = oracle.linear_scan_varlen_bwd(*(np.abs(_np(x)) for x in (a,)), cu,
                                      *(np.abs(_np(x)) for x in (A32, H32, gA, gH)),
                                      None if h0 is None else np.abs(_np(h0)))
    eb = {"da": scaled_error(_np(da), r[0], S[0]), "db": scaled_error(_np(db), r[1], S[1])}
    if h0 is not None:
        eb["dh0"] = scaled_error(_np(dh0), r[2], S[2])
    assert max(eb.values()) <= tol, eb
    mg.workspace_status()
    return {**errs, **eb}


@pytest.mark.parametrize("D", [256, 37])
@pytest.mark.parametrize("with_h0", [True, False])
def test_varlen_ragged(cuda_lib, D, with_h0):
    """Many sequences of 1..700 rows with empty ones among them: boundaries
    fall anywhere inside tiles, rounds and look-back chains."""
    rng = np.random.default_rng(46 + D)
    lens = _lens(rng, 23, 1, 700, empty_every=5)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    a, b, gA, gH = (x[0] for x in wl.mingru_linear(1, int(cu[-1]), D, seed=47))
    h0 = torch.randn(len(lens), D, generator=torch.Generator().manual_seed(48)) if with_h0 else None
    _varlen_case(cuda_lib, a, b, cu, h0, gA, gH, TOL_F32)


def test_varlen_single_row_sequences_and_long_one(cuda_lib):
    lens = [1] * 40 + [5000] + [1, 0, 0, 2] + [3000]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    a, b, gA, gH = (x[0] for x in wl.mingru_linear(1, int(cu[-1]), 64, seed=49))
    h0 = torch.randn(len(lens), 64, generator=torch.Generator().manual_seed(50))
    _varlen_case(cuda_lib, a, b, cu, h0, gA, gH, TOL_F32)


def test_varlen_bf16(cuda_lib):
    rng = np.random.default_rng(51)
    lens = _lens(rng, 9, 50, 900)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    a, b, gA, gH = (x[0] for x in wl.mingru_linear(1, int(cu[-1]), 128, seed=52,
                                                    in_dtype=torch.bfloat16))
    h0 = torch.randn(len(lens), 128, generator=torch.Generator().manual_seed(53))
    _varlen_case(cuda_lib, a, b, cu, h0, gA, gH, TOL_F32)


def test_varlen_uniform_equals_batched_h0(cuda_lib):
    """B sequences of length T packed back to back: the same results as the
    (B,T,D) op from the same start states (to the float32 bar; the tiles
    differ)."""
    mg = cuda_lib
    B, T, D = 4, 900, 128
    a, b, _, _ = wl.mingru_linear(B, T, D, seed=54, device=DEV, grads=False)
    h0 = torch.randn(B, D, device=DEV, generator=torch.Generator(DEV).manual_seed(55))
    A1, H1 = mg.linear_scan_h0_fwd(a, b, h0)
    cu = torch.arange(B + 1, dtype=torch.int64) * T
    A2, H2 = mg.linear_scan_varlen_fwd(a.reshape(B * T, D), b.reshape(B * T, D), cu, h0)
    assert scaled_error(_np(A2).reshape(B, T, D), _np(A1)) <= TOL_F32
    assert scaled_error(_np(H2).reshape(B, T, D), _np(H1), np.abs(_np(H1))) <= 1e-3


def test_varlen_bad_offsets_are_reported(cuda_lib):
    """A decreasing cu_seqlens is detected on the device (no fault), reported
    by the workspace status, and the next valid call is correct."""
    mg = cuda_lib
    a, b, _, _ = (x[0] if x is not None else None
                  for x in wl.mingru_linear(1, 600, 64, seed=56, device=DEV, grads=False))
    ws = mg.new_workspace(mg.varlen_workspace_size(600, 64), DEV)
    bad = torch.tensor([0, 300, 100, 600], dtype=torch.int64)
    mg.linear_scan_varlen_fwd(a, b, bad, ws=ws)
    with pytest.raises(mg.MgScanError) as ei:
        mg.workspace_status(ws)
    assert ei.value.status == mg.MG_ERR_INVALID_ARG
    good = np.array([0, 100, 300, 600], dtype=np.int64)
    A, H = mg.linear_scan_varlen_fwd(a, b, torch.as_tensor(good), ws=ws)
    mg.workspace_status(ws)
    import oracle
    rA, rH = oracle.linear_scan_varlen_fwd(a.cpu(), b.cpu(), good)
    assert scaled_error(_np(A), rA) <= TOL_F32


@pytest.mark.parametrize("case", ["all_empty", "T0_h0"])
def test_varlen_degenerate(cuda_lib, case):
    mg = cuda_lib
    if case == "all_empty":
        e = torch.zeros(0, 8, device=DEV)
        h0 = torch.ones(3, 8, device=DEV)
        A, H = mg.linear_scan_varlen_fwd(e, e, [0, 0, 0, 0], h0)
        assert A.shape == (0, 8)
        da, db, dh0 = mg.linear_scan_varlen_bwd(e, [0, 0, 0, 0], e, e, e, e, h0,
                                                out=(None, None, torch.full((3, 8), 7.0, device=DEV)))
        assert torch.equal(dh0, torch.zeros(3, 8, device=DEV))
    else:
        a = torch.zeros(2, 0, 8, device=DEV)
        h0 = torch.ones(2, 8, device=DEV)
        _, _, dh0 = mg.linear_scan_h0_bwd(a, h0, a, a, a, a,
                                          out=(None, None, torch.full((2, 8), 7.0, device=DEV)))
        assert torch.equal(dh0, torch.zeros(2, 8, device=DEV))


@pytest.mark.parametrize("k,v,shape", [(4, 4, (2, 333, 5)), (2, 8, (2, 200, 3)), (1, 4, (2, 300, 7)),
                                       (4, 16, (1, 700, 3)), (8, 8, (2, 200, 3)),
                                       (16, 16, (2, 150, 3)), (16, 4, (1, 300, 2))])
def test_affine_h0(cuda_lib, k, v, shape):
    """Every kernel family (lane kernel, chunk engine, warp kernel) from a
    start state; the parity metric as for the plain affine ops."""
    import oracle
    from parity import block_rms
    mg = cuda_lib
    Bq, Tq, nq = shape
    A, Bm, gA, gB = wl.haar_affine(Bq, Tq, nq, k, v, seed=57)
    H0 = torch.randn(Bq, nq, k, v, generator=torch.Generator().manual_seed(58))
    Abar, Bbar = mg.affine_scan_h0_fwd(A.to(DEV), Bm.to(DEV), H0.to(DEV),
                                       out=(_nan(A.shape), _nan(Bm.shape)))
    rAbar, rBbar = oracle.affine_scan_h0_fwd(A, Bm, H0)
    if k == 1:
        SA, SB = oracle.affine_scan_h0_fwd(np.abs(_np(A)), np.abs(_np(Bm)), np.abs(_np(H0)))
    else:
        SA, SB = block_rms(rAbar), block_rms(rBbar)
    errs = {"Abar": scaled_error(_np(Abar), rAbar, SA), "Bbar": scaled_error(_np(Bbar), rBbar, SB)}
    assert max(errs.values()) <= TOL_F32, errs
    Ab32, Bb32 = torch.from_numpy(rAbar).float(), torch.from_numpy(rBbar).float()
    dA, dB, dH0 = mg.affine_scan_h0_bwd(A.to(DEV), H0.to(DEV), Ab32.to(DEV), Bb32.to(DEV),
                                        gA.to(DEV), gB.to(DEV),
                                        out=(_nan(A.shape), _nan(Bm.shape), _nan(H0.shape)))
    rdA, rdB, rdH0 = oracle.affine_scan_h0_bwd(A, H0, Ab32, Bb32, gA, gB)
    if k == 1:
        S = oracle.affine_scan_h0_bwd(*(np.abs(_np(x)) for x in (A, H0, Ab32, Bb32, gA, gB)))
    else:
        S = (block_rms(rdA), block_rms(rdB), block_rms(rdH0))
    eb = {"dA": scaled_error(_np(dA), rdA, S[0]), "dB": scaled_error(_np(dB), rdB, S[1]),
          "dH0": scaled_error(_np(dH0), rdH0, S[2])}
    assert max(eb.values()) <= TOL_F32, eb
    mg.workspace_status()


def test_affine_h0_zero_equals_plain_op(cuda_lib):
    mg = cuda_lib
    for k, v in ((4, 4), (16, 16)):
        A, Bm, _, _ = wl.haar_affine(2, 300, 4, k, v, seed=59, device=DEV, grads=False)
        Z = torch.zeros(2, 4, k, v, device=DEV)
        r1 = mg.affine_scan_h0_fwd(A, Bm, Z)
        r0 = mg.affine_scan_fwd(A, Bm)
        assert torch.equal(r1[0], r0[0]) and torch.equal(r1[1], r0[1])
