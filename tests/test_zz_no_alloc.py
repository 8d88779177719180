"""The no-allocation entry point, mg_linear_scan_fwd_noalloc, called through
the C ABI.

Some callers cannot allocate device memory when they call the scan (a plugin
whose host framework gives it no allocator, code that must not allocate once
running).  This entry point takes no workspace: it uses a static scratch array
inside the library.  It runs the same kernel as the regular entry point
mg_linear_scan_fwd (which uses a caller workspace), so the test asks for
bitwise-equal outputs on consecutive calls (two in a row on the same inputs,
and a large -> small -> large sequence of shapes sharing the scratch), checks
one case against the float64 oracle within the parity tolerance, reads the
scratch's device-side status after every call, and checks that a size too
large for the static scratch is refused before any launch.

This file sorts last so that a run stopping at its first failure has already
run every other test; it also passes alone in a fresh process.
"""
from __future__ import annotations

import pytest
import torch

from linear_recurrence_scans_gb300 import workloads as wl
from parity import TOL_BF16, TOL_F32, linear_fwd_errors

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc(mg, a, b):
    lib = mg.load()
    B, T, D = a.shape
    code = mg.MG_F32 if a.dtype == torch.float32 else mg.MG_BF16
    A = torch.full((B, T, D), float("nan"), device=DEV)
    Bc = torch.full((B, T, D), float("nan"), device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    st = lib.mg_linear_scan_fwd_noalloc(a.data_ptr(), b.data_ptr(), code, A.data_ptr(),
                                        Bc.data_ptr(), B, T, D, s)
    assert st == mg.MG_OK, lib.mg_last_error_detail()
    assert lib.mg_linear_scan_fwd_noalloc_status(s) == mg.MG_OK, lib.mg_last_error_detail()
    return A, Bc


def _same_as_workspace_entry_point(mg, a, b):
    A, Bc = _noalloc(mg, a, b)
    ref_A, ref_Bc = mg.linear_scan_fwd(a, b)           # regular entry point, caller workspace
    torch.cuda.synchronize()
    assert torch.equal(A, ref_A) and torch.equal(Bc, ref_Bc)
    return A, Bc


def test_noalloc_matches_workspace_entry_point_and_oracle(cuda_lib):
    mg = cuda_lib
    # large -> small -> large, float32 and bf16: consecutive calls share the scratch
    cases = [((4, 2048, 1024), torch.float32, 41, TOL_F32),
             ((3, 517, 300), torch.float32, 42, TOL_F32),
             ((1, 37, 8), torch.float32, 45, TOL_F32),
             ((2, 700, 512), torch.bfloat16, 43, TOL_BF16),
             ((4, 2048, 1024), torch.float32, 46, TOL_F32)]
    for i, (shape, dtype, seed, tol) in enumerate(cases):
        a, b, _, _ = wl.mingru_linear(*shape, seed=seed, device=DEV, in_dtype=dtype, grads=False)
        A, Bc = _same_as_workspace_entry_point(mg, a, b)
        if i in (1, 3):   # against the float64 oracle as well
            errs = linear_fwd_errors(a.cpu(), b.cpu(), A, Bc)
            assert max(errs.values()) <= tol, (shape, dtype, errs)


def test_noalloc_twice_in_a_row_same_inputs(cuda_lib):
    mg = cuda_lib
    a, b, _, _ = wl.mingru_linear(4, 2048, 1024, seed=44, device=DEV, grads=False)
    first = _same_as_workspace_entry_point(mg, a, b)
    second = _same_as_workspace_entry_point(mg, a, b)
    assert torch.equal(first[0], second[0]) and torch.equal(first[1], second[1])


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
    assert lib.mg_linear_scan_fwd_noalloc_status(torch.cuda.current_stream().cuda_stream) == mg.MG_OK
