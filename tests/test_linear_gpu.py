"""GPU parity of mg_linear_scan_fwd / mg_linear_scan_bwd against the float64
oracle, through the C ABI (via the Python binding)."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from linear_recurrence_scans_gb300 import workloads as wl
from parity import TOL_BF16, TOL_F32, linear_bwd_errors, linear_fwd_errors

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _nan_like(x):
    return torch.full_like(x, float("nan"), dtype=torch.float32)


def _run_fwd_bwd(mg, a, b, gA, gBc, tol):
    """Fwd parity, then bwd parity with the oracle's fwd outputs (rounded to
    float32) as A, Bc on both sides.  Outputs start as NaN so an unwritten
    element fails."""
    ad, bd = a.to(DEV), b.to(DEV)
    A, Bc = mg.linear_scan_fwd(ad, bd, out=(_nan_like(ad), _nan_like(ad)))
    errs = linear_fwd_errors(a, b, A, Bc)
    assert max(errs.values()) <= tol, errs
    import oracle
    rA, rBc = oracle.linear_scan_fwd(a, b)
    A32, Bc32 = torch.from_numpy(rA).float(), torch.from_numpy(rBc).float()
    da, db = mg.linear_scan_bwd(ad, A32.to(DEV), Bc32.to(DEV), gA.to(DEV), gBc.to(DEV),
                                out=(_nan_like(ad), _nan_like(ad)))
    errs_b = linear_bwd_errors(a, A32, Bc32, gA, gBc, da, db)
    assert max(errs_b.values()) <= tol, errs_b
    mg.workspace_status()
    return {**errs, **errs_b}


def test_uniform_2x256x64(cuda_lib):
    """linear_scan_fwd fp32, a ~ U(0,1), b ~ N(0,1), (2,256,64), seed 0."""
    mg = cuda_lib
    a, b = wl.uniform_linear(2, 256, 64, seed=0)
    g = torch.Generator().manual_seed(9)
    gA, gBc = torch.randn(a.shape, generator=g), torch.randn(a.shape, generator=g)
    _run_fwd_bwd(mg, a, b, gA, gBc, TOL_F32)


@pytest.mark.parametrize("shape", [
    (1, 1, 4),        # one step
    (1, 3, 4),        # shorter than a thread's steps
    (3, 517, 300),    # ragged time tail and ragged channel tile (300 = 2*128 + 44)
    (2, 1000, 37),    # D not a multiple of 4: the one-channel-per-thread variant
    (1, 4099, 8),     # many chunks, a single narrow channel tile (deep look-back)
    (5, 129, 1030),   # several channel tiles per batch row, ragged
])
def test_mingru_shapes(cuda_lib, shape):
    a, b, gA, gBc = wl.mingru_linear(*shape, seed=3)
    _run_fwd_bwd(cuda_lib, a, b, gA, gBc, TOL_F32)


def test_signed_coefficients(cuda_lib):
    """a of both signs and above 1 in magnitude (no positivity assumed)."""
    g = torch.Generator().manual_seed(4)
    a = (torch.rand(2, 700, 64, generator=g) * 1.4 - 0.7)
    b = torch.randn(2, 700, 64, generator=g)
    gA, gBc = torch.randn(a.shape, generator=g), torch.randn(a.shape, generator=g)
    _run_fwd_bwd(cuda_lib, a, b, gA, gBc, TOL_F32)


def test_mingru_8x4096x1024_full(cuda_lib):
    """The minGRU-shaped workload at full size, every element checked."""
    a, b, gA, gBc = wl.mingru_linear(8, 4096, 1024, seed=0)
    errs = _run_fwd_bwd(cuda_lib, a, b, gA, gBc, TOL_F32)
    print("mingru_linear_8x4096x1024", errs)


@pytest.mark.parametrize("shape", [(2, 300, 256), (3, 77, 40), (1, 50, 13)])
def test_bf16_inputs(cuda_lib, shape):
    """bf16 a, b (fp32 accumulation, fp32 outputs); the oracle gets the same
    bf16-rounded values widened exactly."""
    mg = cuda_lib
    a, b, gA, gBc = wl.mingru_linear(*shape, seed=5, in_dtype=torch.bfloat16)
    _run_fwd_bwd(mg, a, b, gA, gBc, TOL_BF16)
    # the bf16 path's error is only fp32 accumulation: it also meets the fp32 bar
    _run_fwd_bwd(mg, a, b, gA, gBc, TOL_F32)


def test_bitwise_reproducible(cuda_lib):
    mg = cuda_lib
    a, b, gA, gBc = wl.mingru_linear(4, 3000, 512, seed=6, device=DEV)
    A1, Bc1 = mg.linear_scan_fwd(a, b)
    A2, Bc2 = mg.linear_scan_fwd(a, b)
    assert torch.equal(A1, A2) and torch.equal(Bc1, Bc2)
    d1 = mg.linear_scan_bwd(a, A1, Bc1, gA, gBc)
    d2 = mg.linear_scan_bwd(a, A1, Bc1, gA, gBc)
    assert torch.equal(d1[0], d2[0]) and torch.equal(d1[1], d2[1])


def test_workspace_reuse_across_shapes(cuda_lib):
    """One workspace, sized for the largest call, reused by smaller and
    differently tiled calls without clearing."""
    mg = cuda_lib
    big = (2, 2000, 512)
    ws = mg.new_workspace(mg.linear_workspace_size(*big), DEV)
    for shape in (big, (1, 300, 64), (3, 100, 37), big):
        a, b, gA, gBc = wl.mingru_linear(*shape, seed=7)
        A, Bc = mg.linear_scan_fwd(a.to(DEV), b.to(DEV), ws=ws)
        errs = linear_fwd_errors(a, b, A, Bc)
        assert max(errs.values()) <= TOL_F32, (shape, errs)
        mg.workspace_status(ws)


def test_degenerate_shapes(cuda_lib):
    mg = cuda_lib
    for shape in ((0, 5, 4), (2, 0, 4), (2, 5, 0)):
        a = torch.zeros(shape, device=DEV)
        A, Bc = mg.linear_scan_fwd(a, a)
        assert A.shape == shape and Bc.shape == shape
        da, db = mg.linear_scan_bwd(a, a, a, a, a)
        assert da.shape == shape


def test_c_abi_rejects_misaligned_and_overlapping(cuda_lib):
    mg = cuda_lib
    lib = mg.load()
    a = torch.rand(2, 16, 8, device=DEV)
    out = torch.empty(2, 2, 16, 8, device=DEV)
    ws = mg.new_workspace(mg.linear_workspace_size(2, 16, 8), DEV)
    s = torch.cuda.current_stream().cuda_stream
    st = lib.mg_linear_scan_fwd(a.data_ptr() + 4, a.data_ptr(), 0, out[0].data_ptr(),
                                out[1].data_ptr(), 2, 15, 8, ws.data_ptr(), ws.numel(), s)
    assert st == mg.MG_ERR_INVALID_ARG
    st = lib.mg_linear_scan_fwd(a.data_ptr(), a.data_ptr(), 0, out[0].data_ptr(),
                                out[0].data_ptr() + 64, 2, 16, 8, ws.data_ptr(), ws.numel(), s)
    assert st == mg.MG_ERR_INVALID_ARG
    with pytest.raises(mg.MgScanError):
        mg.linear_scan_fwd(a, a, out=(out[0], out[0]))


@pytest.mark.large
def test_mingru_bf16_16x32768x4096_sampled(cuda_lib):
    """The large bf16 workload (2^31 elements, 64-bit offsets) in the launch
    configuration the bench times.  Channels are independent, so the oracle
    on 256 seeded (b, d) columns over the full T is exact for those columns.
    Forward parity on the columns; backward chained from each side's own
    forward (the GPU bwd consumes the GPU fwd outputs, the oracle its own)."""
    mg = cuda_lib
    B, T, D = 16, 32768, 4096
    a, b, gA, gBc = wl.mingru_linear(B, T, D, seed=0, device=DEV, in_dtype=torch.bfloat16)
    A, Bc = mg.linear_scan_fwd(a, b)
    da, db = mg.linear_scan_bwd(a, A, Bc, gA, gBc)
    torch.cuda.synchronize()
    mg.workspace_status()
    rng = np.random.default_rng(1234)
    flat = rng.choice(B * D, size=256, replace=False)
    # include the extreme channels
    flat[:4] = [0, D - 1, (B - 1) * D, B * D - 1]
    bs = torch.as_tensor(flat // D, device=DEV)
    ds = torch.as_tensor(flat % D, device=DEV)

    def cols(x):  # (B,T,D) -> (1, T, 256) on the host
        return x[bs, :, ds].transpose(0, 1).unsqueeze(0).cpu()

    ca, cb, cgA, cgBc = cols(a), cols(b), cols(gA), cols(gBc)
    errs = linear_fwd_errors(ca, cb, cols(A), cols(Bc))
    assert max(errs.values()) <= TOL_BF16, errs
    import oracle
    rA, rBc = oracle.linear_scan_fwd(ca, cb)
    errs_b = linear_bwd_errors(ca, rA, rBc, cgA, cgBc, cols(da), cols(db))
    assert max(errs_b.values()) <= TOL_BF16, errs_b
    print("mingru_linear_bf16_16x32768x4096 sampled", errs, errs_b)
