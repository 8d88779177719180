"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol the public header declares, sizes workspaces, and rejects bad
arguments before touching the device."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import linear_recurrence_scans_gb300 as mg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(mg_\w+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from linear_recurrence_scans_gb300 import _build
    _build.build()
    return mg.load()


def test_exports_every_declared_symbol(lib):
    declared = _header_functions()
    assert declared, "no functions found in include/*.h"
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(mg.SYMBOLS) <= set(declared)


def test_abi_version_and_strerror(lib):
    assert lib.mg_abi_version() == 1
    for st in range(5):
        assert lib.mg_strerror(st)
    assert lib.mg_strerror(99) == b"unknown status"


def test_workspace_sizes(lib):
    assert mg.linear_workspace_size(8, 4096, 1024) > 256
    assert mg.linear_workspace_size(0, 4096, 1024) == 256
    assert lib.mg_linear_scan_workspace_size(-1, 2, 3) == 0
    assert mg.log_workspace_size(16, 2048, 2048) > 256
    # grows with the problem
    assert mg.linear_workspace_size(8, 8192, 1024) > mg.linear_workspace_size(8, 4096, 1024)


def _fwd(lib, a=None, b=None, dt=0, A=None, Bc=None, B=2, T=3, D=4, ws=None, wsb=0):
    return lib.mg_linear_scan_fwd(a, b, dt, A, Bc, B, T, D, ws, wsb, None)


def test_rejects_bad_arguments_before_launch(lib):
    # unsupported dtype
    assert _fwd(lib, dt=7) == mg.MG_ERR_UNSUPPORTED
    assert b"dtype" in lib.mg_last_error_detail()
    # negative size
    assert _fwd(lib, B=-1) == mg.MG_ERR_INVALID_ARG
    # degenerate sizes: OK, no launch, no pointer needed
    assert _fwd(lib, B=0) == mg.MG_OK
    assert _fwd(lib, T=0) == mg.MG_OK
    assert _fwd(lib, D=0) == mg.MG_OK
    # NULL workspace
    assert _fwd(lib) == mg.MG_ERR_INVALID_ARG
    assert b"workspace" in lib.mg_last_error_detail()
    # Fake, never dereferenced addresses: validation fails before any CUDA call.
    base = 1 << 40
    need = mg.linear_workspace_size(2, 3, 4)
    ws = base + (1 << 20)
    assert _fwd(lib, ws=ws, wsb=need - 1) == mg.MG_ERR_INVALID_ARG  # too small
    assert _fwd(lib, ws=ws + 16, wsb=need) == mg.MG_ERR_INVALID_ARG  # misaligned ws
    assert _fwd(lib, a=base + 4, b=base + 4096, A=base + 8192, Bc=base + 12288,
                ws=ws, wsb=need) == mg.MG_ERR_INVALID_ARG              # misaligned a
    assert b"aligned" in lib.mg_last_error_detail()
    assert _fwd(lib, a=base, b=base + 4096, A=base + 8192, Bc=base + 8192 + 16,
                ws=ws, wsb=need) == mg.MG_ERR_INVALID_ARG              # A overlaps Bc
    assert b"overlaps" in lib.mg_last_error_detail()
    assert _fwd(lib, a=base, b=base + 4096, A=base, Bc=base + 12288,
                ws=ws, wsb=need) == mg.MG_ERR_INVALID_ARG              # in-place A = a
    # affine envelope
    assert lib.mg_affine_scan_fwd(None, None, None, None, 1, 2, 3, 3, 4, None, 0, None) \
        == mg.MG_ERR_UNSUPPORTED
    assert lib.mg_affine_scan_workspace_size(1, 2, 3, 5, 4) == 0
    # log op: T = -1 is invalid, T = 0 is a no-op
    assert lib.mg_log_scan_fwd(None, None, None, 1, -1, 4, None, 0, None) == mg.MG_ERR_INVALID_ARG
    assert lib.mg_log_scan_fwd(None, None, None, 1, 0, 4, None, 0, None) == mg.MG_OK


def test_binding_rejects_cpu_tensors():
    import torch
    with pytest.raises(ValueError):
        mg.linear_scan_fwd(torch.zeros(1, 2, 4), torch.zeros(1, 2, 4))


def test_rejects_channel_counts_beyond_32_bit_indexing(lib):
    """The channel-wise kernels index channels with 32-bit integers: a D at or
    above 2^31 is refused before launch (it would wrap), a D just below the
    limit is not refused for its size."""
    D = 1 << 31
    assert _fwd(lib, B=1, T=1, D=D) == mg.MG_ERR_UNSUPPORTED
    assert b"channels" in lib.mg_last_error_detail()
    assert lib.mg_linear_scan_bwd(None, 0, None, None, None, None, None, None, 1, 1, D,
                                  None, 0, None) == mg.MG_ERR_UNSUPPORTED
    assert lib.mg_log_scan_fwd(None, None, None, 1, 1, D, None, 0, None) == mg.MG_ERR_UNSUPPORTED
    assert lib.mg_log_scan_bwd(None, None, None, None, None, None, 1, 1, D, None, 0,
                               None) == mg.MG_ERR_UNSUPPORTED
    # below the limit: the next check (the NULL workspace) is what fails
    assert _fwd(lib, B=1, T=1, D=(1 << 31) - (1 << 16)) == mg.MG_ERR_INVALID_ARG


def test_noalloc_size_limit_matches_the_workspace_size(lib):
    """Every shape whose workspace fits the static scratch is accepted by the
    size check of mg_linear_scan_fwd_noalloc (without a GPU the call then
    stops at the device query, MG_ERR_LAUNCH, never at the size check), and
    a shape far beyond it is refused for its size."""
    cap = int(lib.mg_linear_scan_fwd_noalloc_max_scratch())
    base = 1 << 40
    for shape in ((1, 1 << 13, 1 << 16), (8, 4096, 1024), (2, 1 << 15, 4096), (3, 517, 300)):
        need = mg.linear_workspace_size(*shape)
        st = lib.mg_linear_scan_fwd_noalloc(base, base + (1 << 36), mg.MG_F32, base + (2 << 36),
                                            base + (3 << 36), *shape, None)
        if need <= cap:
            assert b"static scratch" not in lib.mg_last_error_detail(), shape
            assert st != mg.MG_ERR_INVALID_ARG or b"scratch" not in lib.mg_last_error_detail()
    st = lib.mg_linear_scan_fwd_noalloc(base, base + (1 << 36), mg.MG_F32, base + (2 << 36),
                                        base + (3 << 36), 64, 65536, 4096, None)
    assert st == mg.MG_ERR_INVALID_ARG and b"static scratch" in lib.mg_last_error_detail()
