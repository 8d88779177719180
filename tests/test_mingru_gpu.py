"""GPU parity of the minGRU gate fused into the linear scan
(mg_mingru_scan_fwd / mg_mingru_scan_bwd) and of the linear backward with
bf16 gradients (mg_linear_scan_bwd_bf16_grads), against the float64 oracle,
through the C ABI (via the Python binding).  Outputs start as NaN so an
unwritten element fails."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from linear_recurrence_scans_gb300 import workloads as wl
from parity import (TOL_BF16, TOL_F32, linear_bwd_errors, mingru_bwd_errors,
                    mingru_fwd_errors)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _nan(shape, dtype=torch.float32):
    return torch.full(shape, float("nan"), dtype=dtype, device=DEV)


def _fused(mg, x1, x2, gA, gBc, tol, with_A=True, grad_dtype=torch.float32):
    """Forward parity, then backward parity with the oracle's forward outputs
    (rounded to float32) as A, Bc on both sides."""
    import oracle
    d1, d2 = x1.to(DEV), x2.to(DEV)
    shp = tuple(x1.shape)
    A, Bc = mg.mingru_scan_fwd(d1, d2, want_A=with_A,
                               out=(_nan(shp) if with_A else None, _nan(shp)))
    errs = mingru_fwd_errors(x1, x2, A, Bc)
    assert max(errs.values()) <= tol, errs
    rA, rBc = oracle.mingru_scan_fwd(x1, x2)
    A32, Bc32 = torch.from_numpy(rA).float(), torch.from_numpy(rBc).float()
    gtol = tol if grad_dtype == torch.float32 else TOL_BF16
    for ga in (True, False):
        dx1, dx2 = mg.mingru_scan_bwd(d1, d2, A32.to(DEV) if ga else None, Bc32.to(DEV),
                                      gA.to(DEV) if ga else None, gBc.to(DEV),
                                      grad_dtype=grad_dtype,
                                      out=(_nan(shp, grad_dtype), _nan(shp, grad_dtype)))
        eb = mingru_bwd_errors(x1, x2, A32 if ga else None, Bc32, gA if ga else None, gBc,
                               dx1, dx2)
        assert max(eb.values()) <= gtol, (ga, eb)
        errs.update({f"{k}{'' if ga else '_noGA'}": v for k, v in eb.items()})
    mg.workspace_status()
    return errs


@pytest.mark.parametrize("shape", [
    (1, 1, 4),        # one step
    (1, 3, 8),        # shorter than a thread's steps
    (3, 517, 300),    # ragged time tail and channel tile
    (2, 1000, 37),    # D not a multiple of 4: the one-channel-per-thread variant
    (1, 4099, 8),     # many chunks, one narrow channel tile
    (5, 129, 1030),
])
def test_fused_fp32_shapes(cuda_lib, shape):
    x1, x2, gA, gBc = wl.mingru_x(*shape, seed=31)
    _fused(cuda_lib, x1, x2, gA, gBc, TOL_F32)


def test_fused_fp32_without_A(cuda_lib):
    x1, x2, gA, gBc = wl.mingru_x(2, 700, 256, seed=32)
    _fused(cuda_lib, x1, x2, gA, gBc, TOL_F32, with_A=False)


@pytest.mark.parametrize("shape", [(2, 300, 256), (3, 77, 40), (1, 50, 13)])
def test_fused_bf16_inputs(cuda_lib, shape):
    """bf16 x1, x2 (the oracle gets the same rounded values widened exactly):
    the error is float32 evaluation only, so the float32 bar holds too."""
    x1, x2, gA, gBc = wl.mingru_x(*shape, seed=33, in_dtype=torch.bfloat16)
    _fused(cuda_lib, x1, x2, gA, gBc, TOL_F32)


@pytest.mark.parametrize("shape", [(2, 300, 256), (1, 50, 13)])
def test_fused_bf16_gradients(cuda_lib, shape):
    x1, x2, gA, gBc = wl.mingru_x(*shape, seed=34, in_dtype=torch.bfloat16)
    _fused(cuda_lib, x1, x2, gA, gBc, TOL_F32, grad_dtype=torch.bfloat16)


def test_fused_extreme_gates(cuda_lib):
    """Saturated gates (|x1| up to 60: z rounds to 0 or 1 in float32) and
    large |x2| on both branches of g, including g's branch point 0."""
    g = torch.Generator().manual_seed(35)
    x1 = torch.randn(2, 400, 64, generator=g) * 20
    x2 = torch.randn(2, 400, 64, generator=g) * 10
    x2[:, ::7] = 0.0
    gA, gBc = torch.randn(x1.shape, generator=g), torch.randn(x1.shape, generator=g)
    _fused(cuda_lib, x1, x2, gA, gBc, TOL_F32)


def test_fused_8x4096x1024_full(cuda_lib):
    """The minGRU workload's shape at full size, every element checked."""
    x1, x2, gA, gBc = wl.mingru_x(8, 4096, 1024, seed=0)
    print("mingru fused 8x4096x1024", _fused(cuda_lib, x1, x2, gA, gBc, TOL_F32))


def test_fused_matches_gate_then_scan(cuda_lib):
    """The fused forward against the unfused path on the same inputs: the
    gate computed by torch in float64, rounded to float32, then the linear
    scan op; both within the float32 bar of the oracle, and of each other."""
    mg = cuda_lib
    x1, x2, _, _ = wl.mingru_x(2, 900, 128, seed=36, device=DEV, grads=False)
    A, Bc = mg.mingru_scan_fwd(x1, x2)
    z = torch.sigmoid(x1.double())
    a = torch.sigmoid(-x1.double()).float()
    b = (z * torch.where(x2 >= 0, x2.double() + 0.5, torch.sigmoid(x2.double()))).float()
    A2, Bc2 = mg.linear_scan_fwd(a, b)
    from parity import scaled_error
    assert scaled_error(A.double().cpu().numpy(), A2.double().cpu().numpy()) <= 1e-4
    assert scaled_error(Bc.double().cpu().numpy(), Bc2.double().cpu().numpy(),
                        np.abs(Bc2.double().cpu().numpy())) <= 1e-4


def test_bitwise_reproducible(cuda_lib):
    mg = cuda_lib
    x1, x2, gA, gBc = wl.mingru_x(4, 3000, 512, seed=37, device=DEV)
    r1 = mg.mingru_scan_fwd(x1, x2)
    r2 = mg.mingru_scan_fwd(x1, x2)
    assert torch.equal(r1[0], r2[0]) and torch.equal(r1[1], r2[1])
    d1 = mg.mingru_scan_bwd(x1, x2, r1[0], r1[1], gA, gBc)
    d2 = mg.mingru_scan_bwd(x1, x2, r1[0], r1[1], gA, gBc)
    assert torch.equal(d1[0], d2[0]) and torch.equal(d1[1], d2[1])


def test_fused_rejects_bad_arguments(cuda_lib):
    mg = cuda_lib
    x = torch.zeros(2, 8, 4, device=DEV)
    with pytest.raises(ValueError):
        mg.mingru_scan_bwd(x, x, x, x, None, x)            # A without gA
    lib = mg.load()
    s = torch.cuda.current_stream().cuda_stream
    ws = mg.new_workspace(mg.mingru_workspace_size(2, 8, 4), DEV)
    st = lib.mg_mingru_scan_bwd(x.data_ptr(), x.data_ptr(), 0, None, x.data_ptr(), x.data_ptr(),
                                x.data_ptr(), x.data_ptr(), x.data_ptr(), 0, 2, 8, 4,
                                ws.data_ptr(), ws.numel(), s)
    assert st == mg.MG_ERR_INVALID_ARG                     # gA given, A NULL
    st = lib.mg_mingru_scan_fwd(x.data_ptr(), x.data_ptr(), 5, None, x.data_ptr(), 2, 8, 4,
                                ws.data_ptr(), ws.numel(), s)
    assert st == mg.MG_ERR_UNSUPPORTED                     # dtype


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_linear_bwd_bf16_gradients(cuda_lib, dt):
    """mg_linear_scan_bwd_bf16_grads: the float32 adjoint rounded at the
    store; within the bf16 bar of the oracle, and equal to the float32-output
    op's result rounded to bf16."""
    import oracle
    mg = cuda_lib
    a, b, gA, gBc = wl.mingru_linear(3, 517, 300, seed=38, in_dtype=dt)
    rA, rBc = oracle.linear_scan_fwd(a, b)
    A32, Bc32 = torch.from_numpy(rA).float(), torch.from_numpy(rBc).float()
    args = (a.to(DEV), A32.to(DEV), Bc32.to(DEV), gA.to(DEV), gBc.to(DEV))
    shp = tuple(a.shape)
    da, db = mg.mg_linear_scan_bwd_bf16_grads(*args, out=(_nan(shp, torch.bfloat16),
                                                          _nan(shp, torch.bfloat16)))
    errs = linear_bwd_errors(a, A32, Bc32, gA, gBc, da, db)
    assert max(errs.values()) <= TOL_BF16, errs
    da32, db32 = mg.linear_scan_bwd(*args)
    assert torch.equal(da, da32.to(torch.bfloat16)) and torch.equal(db, db32.to(torch.bfloat16))


@pytest.mark.large
def test_fused_bf16_16x32768x4096_sampled(cuda_lib):
    """The fused op at the large workload's size (2^31 elements, bf16 x1, x2,
    64-bit offsets), in the launch configuration the bench times: forward and
    backward (without gA, as a minGRU layer runs them), checked on 256 seeded
    whole-T channel columns (channels are independent, so the oracle on a
    column is exact for it); the backward consumes the GPU forward's Bc."""
    import oracle
    mg = cuda_lib
    B, T, D = 16, 32768, 4096
    x1, x2, _, gBc = wl.mingru_x(B, T, D, seed=0, device=DEV, in_dtype=torch.bfloat16)
    _, Bc = mg.mingru_scan_fwd(x1, x2, want_A=False)
    dx1, dx2 = mg.mingru_scan_bwd(x1, x2, None, Bc, None, gBc, grad_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    mg.workspace_status()
    rng = np.random.default_rng(4321)
    flat = rng.choice(B * D, size=256, replace=False)
    flat[:4] = [0, D - 1, (B - 1) * D, B * D - 1]
    bs = torch.as_tensor(flat // D, device=DEV)
    ds = torch.as_tensor(flat % D, device=DEV)

    def cols(x):
        return x[bs, :, ds].transpose(0, 1).unsqueeze(0).cpu()

    c1, c2, cg = cols(x1), cols(x2), cols(gBc)
    errs = mingru_fwd_errors(c1, c2, None, cols(Bc))
    assert max(errs.values()) <= TOL_BF16, errs
    _, rBc = oracle.mingru_scan_fwd(c1, c2)
    eb = mingru_bwd_errors(c1, c2, None, rBc, None, cg, cols(dx1), cols(dx2))
    assert max(eb.values()) <= TOL_BF16, eb
    print("mingru fused bf16 16x32768x4096 sampled", errs, eb)
