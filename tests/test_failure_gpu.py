"""Failure detection on the GPU without a GPU fault: a look-back wait that
runs out (its predecessor never publishes) gives up within its bound, the
launch completes, the host reads MG_ERR_TIMEOUT, and the context and the
workspace stay usable.  A workspace that was not zero-filled is reported,
not faulted on."""
from __future__ import annotations

import pytest
import torch

from linear_recurrence_scans_gb300 import workloads as wl
from parity import TOL_F32, linear_fwd_errors

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_stalled_predecessor_times_out_and_recovers(cuda_lib):
    mg = cuda_lib
    lib = mg.load()
    B, T, D = 1, 4096, 128   # one channel tile, many time chunks
    a, b, _, _ = wl.mingru_linear(B, T, D, seed=21, grads=False)
    ad, bd = a.to(DEV), b.to(DEV)
    A, Bc = torch.empty_like(ad), torch.empty_like(ad)
    ws = mg.new_workspace(mg.linear_workspace_size(B, T, D), DEV)
    s = torch.cuda.current_stream().cuda_stream
    st = lib.mg_testing_linear_scan_fwd_stall(ad.data_ptr(), bd.data_ptr(), A.data_ptr(),
                                              Bc.data_ptr(), B, T, D, ws.data_ptr(), ws.numel(),
                                              5, 20_000_000, s)   # tile 5 stalls; 20 ms waits
    assert st == mg.MG_OK
    with pytest.raises(mg.MgScanError) as ei:
        mg.workspace_status(ws)
    assert ei.value.status == mg.MG_ERR_TIMEOUT
    mg.workspace_status(ws)          # the record was cleared
    # the same workspace and context still give correct results
    A2, Bc2 = mg.linear_scan_fwd(ad, bd, ws=ws)
    errs = linear_fwd_errors(a, b, A2, Bc2)
    assert max(errs.values()) <= TOL_F32, errs
    mg.workspace_status(ws)


def test_non_zeroed_workspace_is_reported(cuda_lib):
    mg = cuda_lib
    B, T, D = 2, 700, 64
    a, b, _, _ = wl.mingru_linear(B, T, D, seed=22, grads=False, device=DEV)
    ws = mg.new_workspace(mg.linear_workspace_size(B, T, D), DEV)
    ws.fill_(255)
    mg.linear_scan_fwd(a, b, ws=ws)
    with pytest.raises(mg.MgScanError) as ei:
        mg.workspace_status(ws)
    assert ei.value.status == mg.MG_ERR_INVALID_ARG
    lib = mg.load()
    assert lib.mg_workspace_init(ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream) == 0
    A, Bc = mg.linear_scan_fwd(a, b, ws=ws)
    mg.workspace_status(ws)
    errs = linear_fwd_errors(a.cpu(), b.cpu(), A, Bc)
    assert max(errs.values()) <= TOL_F32, errs


def test_timeout_does_not_poison_later_launches(cuda_lib):
    """A launch that gave up a wait leaves its error record in the workspace.
    Later launches on that workspace, run WITHOUT reading the record first,
    must still wait normally and give correct results; the next status read
    reports the one timeout, once."""
    mg = cuda_lib
    lib = mg.load()
    B, T, D = 1, 4096, 128
    a, b, _, _ = wl.mingru_linear(B, T, D, seed=23, grads=False)
    ad, bd = a.to(DEV), b.to(DEV)
    A, Bc = torch.empty_like(ad), torch.empty_like(ad)
    ws = mg.new_workspace(mg.linear_workspace_size(B, T, D), DEV)
    s = torch.cuda.current_stream().cuda_stream
    st = lib.mg_testing_linear_scan_fwd_stall(ad.data_ptr(), bd.data_ptr(), A.data_ptr(),
                                              Bc.data_ptr(), B, T, D, ws.data_ptr(), ws.numel(),
                                              3, 20_000_000, s)   # tile 3 stalls; 20 ms waits
    assert st == mg.MG_OK
    for _ in range(2):   # no status read in between
        A2, Bc2 = mg.linear_scan_fwd(ad, bd, ws=ws)
        errs = linear_fwd_errors(a, b, A2, Bc2)
        assert max(errs.values()) <= TOL_F32, errs
    with pytest.raises(mg.MgScanError) as ei:
        mg.workspace_status(ws)
    assert ei.value.status == mg.MG_ERR_TIMEOUT
    mg.workspace_status(ws)          # reported once, then cleared


def test_small_then_large_tile_count_on_one_workspace(cuda_lib):
    """The flags of a launch with many tiles lie where an earlier launch with
    few tiles (or another op) kept its data records; the flag tag keeps those
    stale records from reading as flags."""
    from parity import affine_fwd_errors
    mg = cuda_lib
    big = (2, 4000, 512)
    ws = mg.new_workspace(max(mg.linear_workspace_size(*big),
                              mg.affine_workspace_size(2, 300, 4, 4, 4)), DEV)
    Am, Bm, _, _ = wl.haar_affine(2, 300, 4, 4, 4, seed=24)
    Abar, Bbar = mg.affine_scan_fwd(Am.to(DEV), Bm.to(DEV), ws=ws)
    errs = affine_fwd_errors(Am, Bm, Abar, Bbar)
    assert max(errs.values()) <= TOL_F32, errs
    for shape in ((1, 64, 8), big):
        a, b, _, _ = wl.mingru_linear(*shape, seed=25)
        A, Bc = mg.linear_scan_fwd(a.to(DEV), b.to(DEV), ws=ws)
        errs = linear_fwd_errors(a, b, A, Bc)
        assert max(errs.values()) <= TOL_F32, (shape, errs)
    mg.workspace_status(ws)


def test_prefix_words_of_an_earlier_launch_are_not_taken(cuda_lib):
    """A chunk takes its predecessor's prefix record without the flag when
    every word carries the running launch's tag.  Launches on one workspace
    with the same shape but different inputs leave the previous launch's
    words in place: each launch must still match the oracle on its own
    inputs (a stale word accepted would carry the earlier inputs' prefix)."""
    from parity import log_fwd_errors
    mg = cuda_lib
    shape = (2, 4096, 256)   # 2 x 2 channel tiles, dozens of chunks each
    ws = mg.new_workspace(max(mg.linear_workspace_size(*shape), mg.log_workspace_size(*shape)),
                          DEV)
    for seed in (31, 32, 33):
        a, b, _, _ = wl.mingru_linear(*shape, seed=seed, grads=False)
        A, Bc = mg.linear_scan_fwd(a.to(DEV), b.to(DEV), ws=ws)
        errs = linear_fwd_errors(a, b, A, Bc)
        assert max(errs.values()) <= TOL_F32, (seed, errs)
        mg.workspace_status(ws)
    for seed in (34, 35):
        lc, lv = wl.mingru_log(*shape, seed=seed)
        h = mg.parallel_scan_log_fwd(lc.to(DEV), lv.to(DEV), ws=ws)
        errs = log_fwd_errors(lc, lv, h)
        assert max(errs.values()) <= TOL_F32, (seed, errs)
        mg.workspace_status(ws)
