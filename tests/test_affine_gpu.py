"""GPU parity of mg_affine_scan_fwd / mg_affine_scan_bwd against the float64
oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from linear_recurrence_scans_gb300 import workloads as wl
from parity import TOL_F32, affine_bwd_errors, affine_fwd_errors

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _nan(x):
    return torch.full(x.shape, float("nan"), device=x.device)


def _run(mg, A, Bm, gAbar, gBbar, tol=TOL_F32):
    """Fwd parity; bwd parity with the oracle's forward outputs (rounded to
    float32) as Abar, Bbar on both sides.  Outputs start as NaN."""
    Ad, Bd = A.to(DEV), Bm.to(DEV)
    Abar, Bbar = mg.affine_scan_fwd(Ad, Bd, out=(_nan(Ad), _nan(Bd)))
    errs = affine_fwd_errors(A, Bm, Abar, Bbar)
    assert max(errs.values()) <= tol, errs
    import oracle
    rAbar, rBbar = oracle.affine_scan_fwd(A, Bm)
    Ab32, Bb32 = torch.from_numpy(rAbar).float(), torch.from_numpy(rBbar).float()
    dA, dB = mg.affine_scan_bwd(Ad, Ab32.to(DEV), Bb32.to(DEV), gAbar.to(DEV), gBbar.to(DEV),
                                out=(_nan(Ad), _nan(Bd)))
    errs_b = affine_bwd_errors(A, Ab32, Bb32, gAbar, gBbar, dA, dB)
    assert max(errs_b.values()) <= tol, errs_b
    mg.workspace_status()
    return {**errs, **errs_b}


KV = [(k, v) for k in (1, 2, 4, 8, 16) for v in (1, 2, 4, 8, 16)]


@pytest.mark.parametrize("k,v", KV)
def test_every_k_v(cuda_lib, k, v):
    """Every supported (k, v), ragged time (several chunks plus a tail)."""
    A, Bm, gA, gB = wl.haar_affine(2, 45, 3, k, v, seed=k * 100 + v)
    _run(cuda_lib, A, Bm, gA, gB)


@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 3, 2), (2, 333, 5), (1, 700, 1)])
@pytest.mark.parametrize("k", [4, 8, 16])
def test_shapes(cuda_lib, shape, k):
    A, Bm, gA, gB = wl.haar_affine(*shape, k, k, seed=7)
    _run(cuda_lib, A, Bm, gA, gB)


@pytest.mark.parametrize("k,v,shape", [
    (2, 2, (2, 600, 37)),   # lane kernel, 5 chunks, a full and a 5-sequence block
    (2, 16, (1, 300, 33)),
    (4, 1, (2, 400, 40)),
    (4, 8, (1, 300, 64)),
    (4, 16, (1, 200, 35)),  # k=4, v=16 stays on the chunk engine
    (1, 4, (2, 300, 45)),
])
def test_multichunk_ragged_blocks(cuda_lib, k, v, shape):
    """Several chunks in time and a ragged last block of sequences for the
    k <= 4 kernels (the look-back and the partial-block copies)."""
    A, Bm, gA, gB = wl.haar_affine(*shape, k, v, seed=k * 10 + v)
    _run(cuda_lib, A, Bm, gA, gB)


def test_general_matrices(cuda_lib):
    """Non-orthogonal transitions with entries of both signs."""
    g = torch.Generator().manual_seed(8)
    for k, v in ((4, 4), (16, 16), (8, 2)):
        A = torch.randn(2, 60, 3, k, k, generator=g) * (0.9 / np.sqrt(k))
        Bm = torch.randn(2, 60, 3, k, v, generator=g)
        gA = torch.randn(A.shape, generator=g)
        gB = torch.randn(Bm.shape, generator=g)
        _run(cuda_lib, A, Bm, gA, gB)


def test_haar_4x2048x64_k4v4_full(cuda_lib):
    A, Bm, gA, gB = wl.haar_affine(4, 2048, 64, 4, 4, seed=0)
    print("haar_affine_4x2048x64_k4v4", _run(cuda_lib, A, Bm, gA, gB))


def test_haar_2x1024x32_k16v16_full(cuda_lib):
    A, Bm, gA, gB = wl.haar_affine(2, 1024, 32, 16, 16, seed=0)
    print("haar_affine_2x1024x32_k16v16", _run(cuda_lib, A, Bm, gA, gB))


def test_orthogonal_invariant_on_gpu(cuda_lib):
    """Abar_t^T Abar_t = 0.95^(2t) I holds for the GPU result too (relative to
    the scale 0.95^(2t), while it stays in float32 normal range)."""
    A, Bm, _, _ = wl.haar_affine(1, 600, 4, 16, 16, seed=9, grads=False)
    Abar, _ = cuda_lib.affine_scan_fwd(A.to(DEV), Bm.to(DEV))
    Ab = Abar.double().cpu()
    G = torch.einsum("tnij,tnil->tnjl", Ab[0], Ab[0])
    scale = 0.95 ** (2 * torch.arange(1, 601, dtype=torch.float64))
    err = (G - scale[:, None, None, None] * torch.eye(16, dtype=torch.float64)).abs().amax(dim=(1, 2, 3))
    assert torch.all(err <= 1e-4 * scale), float((err / scale).max())


def test_bitwise_reproducible(cuda_lib):
    for k in (4, 16):
        A, Bm, gA, gB = wl.haar_affine(2, 1000, 8, k, k, seed=10, device=DEV)
        r1 = cuda_lib.affine_scan_fwd(A, Bm)
        r2 = cuda_lib.affine_scan_fwd(A, Bm)
        assert torch.equal(r1[0], r2[0]) and torch.equal(r1[1], r2[1])
        d1 = cuda_lib.affine_scan_bwd(A, r1[0], r1[1], gA, gB)
        d2 = cuda_lib.affine_scan_bwd(A, r1[0], r1[1], gA, gB)
        assert torch.equal(d1[0], d2[0]) and torch.equal(d1[1], d2[1])
