"""The no-allocation entry point, mg_linear_scan_fwd_noalloc, called through
the C ABI.

Some callers cannot allocate device memory when they call the scan (a plugin
whose host framework gives it no allocator, code that must not allocate once
running).  This entry point takes no workspace: it uses a static scratch array
inside the library.  The test checks that it gives the same results as the
regular entry point mg_linear_scan_fwd (which uses a caller workspace),
within the parity tolerance, on two calls in a row, and that a size too large
for the static scratch is refused before any launch.

This file sorts last so that a run stopping at its first failure has already
run every other test; it also passes alone in a fresh process.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from linear_recurrence_scans_gb300 import workloads as wl
from parity import TOL_BF16, TOL_F32, scaled_error

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _scale(a, b):
    """Componentwise condition scale of Bc (the oracle on |a|, |b|)."""
    import oracle
    return oracle.linear_scan_fwd(a.abs().cpu(), b.abs().cpu())[1]


def _noalloc(lib, a, b, dtype_code):
    B, T, D = a.shape
    A = torch.full((B, T, D), float("nan"), device=DEV)
    Bc = torch.full((B, T, D), float("nan"), device=DEV)
    st = lib.mg_linear_scan_fwd_noalloc(a.data_ptr(), b.data_ptr(), dtype_code, A.data_ptr(),
                                        Bc.data_ptr(), B, T, D,
                                        torch.cuda.current_stream().cuda_stream)
    return st, A, Bc


def test_noalloc_matches_workspace_entry_point(cuda_lib):
    mg = cuda_lib
    lib = mg.load()
    cases = [((2, 1000, 256), torch.float32, 41, TOL_F32),
             ((3, 517, 300), torch.float32, 42, TOL_F32),
             ((2, 700, 512), torch.bfloat16, 43, TOL_BF16)]
    for shape, dtype, seed, tol in cases:   # consecutive calls share the scratch
        a, b, _, _ = wl.mingru_linear(*shape, seed=seed, device=DEV, in_dtype=dtype, grads=False)
        ref_A, ref_Bc = mg.linear_scan_fwd(a, b)            # regular entry point
        code = mg.MG_F32 if dtype == torch.float32 else mg.MG_BF16
        st, A, Bc = _noalloc(lib, a, b, code)
        assert st == mg.MG_OK, lib.mg_last_error_detail()
        torch.cuda.synchronize()
        S = _scale(a.float(), b.float())
        eA = scaled_error(A.double().cpu().numpy(), ref_A.double().cpu().numpy())
        eB = scaled_error(Bc.double().cpu().numpy(), ref_Bc.double().cpu().numpy(), S)
        assert eA <= tol and eB <= tol, (shape, dtype, eA, eB)


def test_noalloc_twice_in_a_row_same_inputs(cuda_lib):
    mg = cuda_lib
    lib = mg.load()
    a, b, _, _ = wl.mingru_linear(4, 2048, 1024, seed=44, device=DEV, grads=False)
    ref_A, ref_Bc = mg.linear_scan_fwd(a, b)
    S = _scale(a, b)
    for _ in range(2):
        st, A, Bc = _noalloc(lib, a, b, mg.MG_F32)
        assert st == mg.MG_OK, lib.mg_last_error_detail()
        torch.cuda.synchronize()
        assert scaled_error(A.double().cpu().numpy(), ref_A.double().cpu().numpy()) <= TOL_F32
        assert scaled_error(Bc.double().cpu().numpy(), ref_Bc.double().cpu().numpy(), S) <= TOL_F32


def test_noalloc_refuses_sizes_beyond_the_scratch(cuda_lib):
    mg = cuda_lib
    lib = mg.load()
    cap = int(lib.mg_linear_scan_fwd_noalloc_max_scratch())
    assert cap == 32 << 20
    B, T, D = 64, 65536, 4096       # far beyond the static scratch; nothing is launched
    base = 1 << 40                  # never dereferenced: refused before any device access
    st = lib.mg_linear_scan_fwd_noalloc(base, base + (1 << 36), mg.MG_F32, base + (2 << 36),
                                        base + (3 << 36), B, T, D, 0)
    assert st == mg.MG_ERR_INVALID_ARG
    assert b"static scratch" in lib.mg_last_error_detail()
