"""GB300-native (sm_103a) minGRU scan family: Python binding of ``libmgscan.so``.

The functions below marshal torch CUDA tensors into the C ABI declared in
``include/mg_scan.h`` and nothing more: every step of every op runs in the
library's CUDA kernels.  torch is used only for device memory and the current
stream.  There is no fallback: if the library is missing or a call fails, an
exception is raised.

Ops (names of the C entry points; aliases with the names of the page
"minGRU - Triton kernels" follow them):

* ``mg_linear_scan_fwd(a, b)              -> (A, Bc)``       alias ``linear_scan_fwd``
* ``mg_linear_scan_bwd(a, A, Bc, gA, gBc) -> (da, db)``      alias ``linear_scan_bwd``
* ``mg_log_scan_fwd(log_coeffs, log_values) -> h``           alias ``parallel_scan_log_fwd``
* ``mg_log_scan_bwd(log_coeffs, log_values, h, gh) -> (dlog_coeffs, dlog_values)``
  alias ``parallel_scan_log_bwd`` (the adjoint of the log-space scan)
* ``mg_affine_scan_fwd(A, Bm)             -> (Abar, Bbar)``  alias ``affine_scan_fwd``
* ``mg_affine_scan_bwd(A, Abar, Bbar, gAbar, gBbar) -> (dA, dB)``  alias ``affine_scan_bwd``
* ``mg_linear_scan_bwd_bf16_grads(a, A, Bc, gA, gBc) -> (da, db)`` (bf16 gradients)
* ``mg_mingru_scan_fwd(x1, x2) -> (A, Bc)`` and ``mg_mingru_scan_bwd(x1, x2, A, Bc, gA, gBc)
  -> (dx1, dx2)``: the minGRU gate fused into the linear scan (aliases
  ``mingru_scan_fwd``, ``mingru_scan_bwd``)
* ``mg_linear_scan_h0_fwd(a, b, h0) -> (A, H)``, ``mg_linear_scan_h0_bwd(a, h0, A, H, gA, gH)
  -> (da, db, dh0)``: the linear scan from start states h0 (B, D)
* ``mg_linear_scan_varlen_fwd(a, b, cu_seqlens, h0=None) -> (A, H)`` and
  ``mg_linear_scan_varlen_bwd(a, cu_seqlens, A, H, gA, gH, h0=None) -> (da, db, dh0)``:
  packed variable-length sequences (Ttot, D) with int64 offsets
* ``mg_affine_scan_h0_fwd(A, Bm, H0) -> (Abar, Bbar)``, ``mg_affine_scan_h0_bwd(A, H0, Abar,
  Bbar, gAbar, gBbar) -> (dA, dB, dH0)``: the affine scan from start states H0 (B, n, k, v)
* ``mg_angle_scan_fwd(theta, scale, gamma, b, h0, perm, sgn, p2p=None) -> h`` and
  ``mg_angle_scan_bwd(...) -> (dtheta, dscale, dgamma, db, dh0)``: the angle-fused
  scan (aliases ``angle_scan_fwd``, ``angle_scan_bwd``)

Every op accepts optional preallocated outputs (``out=(...)``), a workspace
tensor (``ws=``, uint8, zero-filled before first use) and a stream
(``stream=``, a ``torch.cuda.Stream``); by default outputs are allocated with
``torch.empty``, a cached per-(device, stream) workspace is used and the call
is issued on the current stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

__all__ = [
    "MgScanError", "load", "library_path",
    "mg_linear_scan_fwd", "mg_linear_scan_bwd", "mg_log_scan_fwd", "mg_log_scan_bwd",
    "mg_affine_scan_fwd", "mg_affine_scan_bwd",
    "linear_scan_fwd", "linear_scan_bwd", "parallel_scan_log_fwd", "parallel_scan_log_bwd",
    "affine_scan_fwd", "affine_scan_bwd",
    "linear_workspace_size", "log_workspace_size", "affine_workspace_size",
    "workspace_status", "new_workspace",
    "mg_linear_scan_bwd_bf16_grads", "mg_mingru_scan_fwd", "mg_mingru_scan_bwd",
    "mingru_workspace_size", "mingru_scan_fwd", "mingru_scan_bwd",
    "mg_linear_scan_h0_fwd", "mg_linear_scan_h0_bwd", "mg_linear_scan_varlen_fwd",
    "mg_linear_scan_varlen_bwd", "varlen_workspace_size",
    "mg_affine_scan_h0_fwd", "mg_affine_scan_h0_bwd",
    "mg_angle_scan_fwd", "mg_angle_scan_bwd", "angle_scan_fwd", "angle_scan_bwd",
]

MG_OK, MG_ERR_INVALID_ARG, MG_ERR_UNSUPPORTED, MG_ERR_LAUNCH, MG_ERR_TIMEOUT = range(5)
MG_F32, MG_BF16 = 0, 1

SYMBOLS = (
    "mg_abi_version", "mg_strerror", "mg_last_error_detail",
    "mg_linear_scan_workspace_size", "mg_log_scan_workspace_size",
    "mg_affine_scan_workspace_size", "mg_workspace_init", "mg_workspace_status",
    "mg_linear_scan_fwd", "mg_linear_scan_bwd", "mg_log_scan_fwd", "mg_log_scan_bwd",
    "mg_affine_scan_fwd", "mg_affine_scan_bwd",
    "mg_linear_scan_bwd_bf16_grads", "mg_mingru_scan_workspace_size",
    "mg_mingru_scan_fwd", "mg_mingru_scan_bwd",
    "mg_linear_scan_h0_fwd", "mg_linear_scan_h0_bwd", "mg_linear_scan_varlen_workspace_size",
    "mg_linear_scan_varlen_fwd", "mg_linear_scan_varlen_bwd",
    "mg_affine_scan_h0_fwd", "mg_affine_scan_h0_bwd",
    "mg_angle_scan_fwd", "mg_angle_scan_bwd",
)


class MgScanError(RuntimeError):
    """A failed call into libmgscan; ``status`` is the mg_status code."""

    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    """The in-tree build, or the library named by MGSCAN_LIBRARY (another
    build of the same sources, e.g. with different tile sizes)."""
    return os.environ.get("MGSCAN_LIBRARY") or _build.LIB_PATH


def load():
    """Load ``libmgscan.so`` (built by ``__graft_entry__.build()`` or
    ``python -m linear_recurrence_scans_gb300._build``).  Raises if missing."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first "
                               "(python -m linear_recurrence_scans_gb300._build)")
        lib = ctypes.CDLL(path)
        vp, i64, sz, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
        st = ctypes.c_int
        lib.mg_abi_version.argtypes, lib.mg_abi_version.restype = [], i32
        lib.mg_strerror.argtypes, lib.mg_strerror.restype = [st], ctypes.c_char_p
        lib.mg_last_error_detail.argtypes, lib.mg_last_error_detail.restype = [], ctypes.c_char_p
        lib.mg_linear_scan_workspace_size.argtypes = [i64, i64, i64]
        lib.mg_log_scan_workspace_size.argtypes = [i64, i64, i64]
        lib.mg_affine_scan_workspace_size.argtypes = [i64, i64, i64, i32, i32]
        for f in (lib.mg_linear_scan_workspace_size, lib.mg_log_scan_workspace_size,
                  lib.mg_affine_scan_workspace_size):
            f.restype = sz
        lib.mg_workspace_init.argtypes = [vp, sz, vp]
        lib.mg_workspace_status.argtypes = [vp, vp]
        lib.mg_linear_scan_fwd.argtypes = [vp, vp, i32, vp, vp, i64, i64, i64, vp, sz, vp]
        lib.mg_linear_scan_bwd.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, i64, i64, i64, vp, sz, vp]
        lib.mg_log_scan_fwd.argtypes = [vp, vp, vp, i64, i64, i64, vp, sz, vp]
        lib.mg_log_scan_bwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, vp, sz, vp]
        lib.mg_affine_scan_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, i32, vp, sz, vp]
        lib.mg_affine_scan_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, i32,
                                           vp, sz, vp]
        lib.mg_linear_scan_bwd_bf16_grads.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, i64, i64,
                                                      i64, vp, sz, vp]
        lib.mg_mingru_scan_workspace_size.argtypes = [i64, i64, i64]
        lib.mg_mingru_scan_workspace_size.restype = sz
        lib.mg_mingru_scan_fwd.argtypes = [vp, vp, i32, vp, vp, i64, i64, i64, vp, sz, vp]
        lib.mg_mingru_scan_bwd.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, i32, i64, i64, i64,
                                           vp, sz, vp]
        lib.mg_linear_scan_h0_fwd.argtypes = [vp, vp, i32, vp, vp, vp, i64, i64, i64, vp, sz, vp]
        lib.mg_linear_scan_h0_bwd.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64,
                                              i64, vp, sz, vp]
        lib.mg_linear_scan_varlen_workspace_size.argtypes = [i64, i64]
        lib.mg_linear_scan_varlen_workspace_size.restype = sz
        lib.mg_linear_scan_varlen_fwd.argtypes = [vp, vp, i32, vp, i64, vp, vp, vp, i64, i64, vp,
                                                  sz, vp]
        lib.mg_linear_scan_varlen_bwd.argtypes = [vp, i32, vp, i64, vp, vp, vp, vp, vp, vp, vp,
                                                  vp, i64, i64, vp, sz, vp]
        lib.mg_affine_scan_h0_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, vp, sz,
                                              vp]
        lib.mg_affine_scan_h0_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64,
                                              i32, i32, vp, sz, vp]
        lib.mg_angle_scan_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, i64, i64,
                                          i64, i32, i32, vp]
        lib.mg_angle_scan_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, vp,
                                          vp, vp, i64, i64, i64, i32, i32, vp]
        lib.mg_testing_linear_scan_fwd_stall.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, sz,
                                                         i64, ctypes.c_uint64, vp]
        lib.mg_testing_linear_scan_fwd_stall.restype = st
        lib.mg_linear_scan_fwd_noalloc.argtypes = [vp, vp, i32, vp, vp, i64, i64, i64, vp]
        lib.mg_linear_scan_fwd_noalloc.restype = st
        lib.mg_linear_scan_fwd_noalloc_max_scratch.argtypes = []
        lib.mg_linear_scan_fwd_noalloc_max_scratch.restype = sz
        lib.mg_linear_scan_fwd_noalloc_status.argtypes = [vp]
        lib.mg_linear_scan_fwd_noalloc_status.restype = st
        for name in ("mg_workspace_init", "mg_workspace_status", "mg_linear_scan_fwd",
                     "mg_linear_scan_bwd", "mg_log_scan_fwd", "mg_log_scan_bwd",
                     "mg_affine_scan_fwd", "mg_affine_scan_bwd", "mg_linear_scan_bwd_bf16_grads",
                     "mg_mingru_scan_fwd", "mg_mingru_scan_bwd", "mg_linear_scan_h0_fwd",
                     "mg_linear_scan_h0_bwd", "mg_linear_scan_varlen_fwd",
                     "mg_linear_scan_varlen_bwd", "mg_affine_scan_h0_fwd",
                     "mg_affine_scan_h0_bwd", "mg_angle_scan_fwd", "mg_angle_scan_bwd"):
            getattr(lib, name).restype = st
        _lib = lib
    return _lib


def _check(status: int, what: str):
    if status != MG_OK:
        lib = load()
        msg = lib.mg_strerror(status).decode()
        detail = lib.mg_last_error_detail().decode()
        raise MgScanError(status, f"{what}: {msg}" + (f" ({detail})" if detail else ""))


# ---------------------------------------------------------------- workspace

def linear_workspace_size(B: int, T: int, D: int) -> int:
    return int(load().mg_linear_scan_workspace_size(B, T, D))


def log_workspace_size(B: int, T: int, D: int) -> int:
    return int(load().mg_log_scan_workspace_size(B, T, D))


def affine_workspace_size(B: int, T: int, n: int, k: int, v: int) -> int:
    return int(load().mg_affine_scan_workspace_size(B, T, n, k, v))


def mingru_workspace_size(B: int, T: int, D: int) -> int:
    return int(load().mg_mingru_scan_workspace_size(B, T, D))


def varlen_workspace_size(Ttot: int, D: int) -> int:
    return int(load().mg_linear_scan_varlen_workspace_size(Ttot, D))


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-filled uint8 device buffer usable as a workspace."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


_ws_cache: dict = {}


def _stream_handle(stream, device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return int(s.cuda_stream)


def _workspace(nbytes: int, device, stream_handle: int, ws):
    if ws is not None:
        if ws.device != device or ws.dtype != torch.uint8 or not ws.is_contiguous():
            raise ValueError("ws must be a contiguous uint8 tensor on the op's device")
        return ws
    key = (device.index, stream_handle)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        if buf is not None:
            # Kernels on the op's stream (which torch's allocator does not
            # track for this buffer) may still use the smaller workspace:
            # let them finish before it can be freed and reused.
            torch.cuda.synchronize(device)
        # Zero-filled on the current stream; wait for it so that the op's
        # stream (possibly another one) sees a cleared workspace.
        buf = new_workspace(int(nbytes * 1.25) + 4096, device)
        torch.cuda.current_stream(device).synchronize()
        _ws_cache[key] = buf
    return buf


def workspace_status(ws: torch.Tensor | None = None, stream=None) -> None:
    """Raise MgScanError(MG_ERR_TIMEOUT) if a look-back wait gave up on ``ws``
    (default: every cached workspace) since the last check."""
    bufs = [ws] if ws is not None else list(_ws_cache.values())
    for b in bufs:
        _check(load().mg_workspace_status(b.data_ptr(), _stream_handle(stream, b.device)),
               "mg_workspace_status")


# ---------------------------------------------------------------- helpers

def _prep(x: torch.Tensor, name: str, dtypes=(torch.float32,)) -> torch.Tensor:
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if x.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {x.dtype} not in {dtypes}")
    x = x.contiguous()
    if x.data_ptr() % 16:
        x = x.clone()
    return x


def _out(out, i, shape, like, dtype=torch.float32):
    if out is not None and out[i] is not None:
        o = out[i]
        if tuple(o.shape) != tuple(shape) or o.dtype != dtype or not o.is_contiguous() \
                or o.device != like.device:
            raise ValueError(f"out[{i}] must be a contiguous {dtype} tensor of shape {tuple(shape)}")
        return o
    return torch.empty(shape, dtype=dtype, device=like.device)


_DT = {torch.float32: MG_F32, torch.bfloat16: MG_BF16}


# ---------------------------------------------------------------- ops

def mg_linear_scan_fwd(a, b, *, out=None, ws=None, stream=None):
    """(A, Bc), float32 (B,T,D): A_t = a_t A_{t-1}, Bc_t = a_t Bc_{t-1} + b_t.
    a, b: (B,T,D), both float32 or both bf16."""
    a = _prep(a, "a", (torch.float32, torch.bfloat16))
    b = _prep(b, "b", (a.dtype,))
    if a.dim() != 3 or b.shape != a.shape:
        raise ValueError("a and b must both be (B, T, D)")
    B, T, D = a.shape
    A, Bc = _out(out, 0, a.shape, a), _out(out, 1, a.shape, a)
    sh = _stream_handle(stream, a.device)
    w = _workspace(linear_workspace_size(B, T, D), a.device, sh, ws)
    _check(load().mg_linear_scan_fwd(a.data_ptr(), b.data_ptr(), _DT[a.dtype], A.data_ptr(),
                                     Bc.data_ptr(), B, T, D, w.data_ptr(), w.numel(), sh),
           "mg_linear_scan_fwd")
    return A, Bc


def mg_linear_scan_bwd(a, A, Bc, gA, gBc, *, out=None, ws=None, stream=None):
    """(da, db), float32 (B,T,D): grads of sum(gA*A) + sum(gBc*Bc) w.r.t. a, b.
    a: float32 or bf16; A, Bc, gA, gBc: float32, all (B,T,D)."""
    a = _prep(a, "a", (torch.float32, torch.bfloat16))
    A, Bc, gA, gBc = (_prep(x, n) for x, n in ((A, "A"), (Bc, "Bc"), (gA, "gA"), (gBc, "gBc")))
    if a.dim() != 3 or any(x.shape != a.shape for x in (A, Bc, gA, gBc)):
        raise ValueError("a, A, Bc, gA, gBc must all be (B, T, D)")
    B, T, D = a.shape
    da, db = _out(out, 0, a.shape, a), _out(out, 1, a.shape, a)
    sh = _stream_handle(stream, a.device)
    w = _workspace(linear_workspace_size(B, T, D), a.device, sh, ws)
    _check(load().mg_linear_scan_bwd(a.data_ptr(), _DT[a.dtype], A.data_ptr(), Bc.data_ptr(),
                                     gA.data_ptr(), gBc.data_ptr(), da.data_ptr(), db.data_ptr(),
                                     B, T, D, w.data_ptr(), w.numel(), sh),
           "mg_linear_scan_bwd")
    return da, db


def mg_linear_scan_bwd_bf16_grads(a, A, Bc, gA, gBc, *, out=None, ws=None, stream=None):
    """(da, db), bf16 (B,T,D): mg_linear_scan_bwd with the gradients rounded
    to bf16.  a: float32 or bf16; A, Bc, gA, gBc: float32."""
    a = _prep(a, "a", (torch.float32, torch.bfloat16))
    A, Bc, gA, gBc = (_prep(x, n) for x, n in ((A, "A"), (Bc, "Bc"), (gA, "gA"), (gBc, "gBc")))
    if a.dim() != 3 or any(x.shape != a.shape for x in (A, Bc, gA, gBc)):
        raise ValueError("a, A, Bc, gA, gBc must all be (B, T, D)")
    B, T, D = a.shape
    da = _out(out, 0, a.shape, a, torch.bfloat16)
    db = _out(out, 1, a.shape, a, torch.bfloat16)
    sh = _stream_handle(stream, a.device)
    w = _workspace(linear_workspace_size(B, T, D), a.device, sh, ws)
    _check(load().mg_linear_scan_bwd_bf16_grads(a.data_ptr(), _DT[a.dtype], A.data_ptr(),
                                                Bc.data_ptr(), gA.data_ptr(), gBc.data_ptr(),
                                                da.data_ptr(), db.data_ptr(), B, T, D,
                                                w.data_ptr(), w.numel(), sh),
           "mg_linear_scan_bwd_bf16_grads")
    return da, db


def mg_linear_scan_h0_fwd(a, b, h0, *, out=None, ws=None, stream=None):
    """(A, H) float32 (B,T,D): the linear scan of a, b (float32 or bf16) from
    the start states h0 (B, D) float32: H_t = a_t H_{t-1} + b_t, H_0 = h0."""
    a = _prep(a, "a", (torch.float32, torch.bfloat16))
    b = _prep(b, "b", (a.dtype,))
    h0 = _prep(h0, "h0")
    if a.dim() != 3 or b.shape != a.shape or tuple(h0.shape) != (a.shape[0], a.shape[2]):
        raise ValueError("a, b must be (B, T, D) and h0 (B, D)")
    B, T, D = a.shape
    A, H = _out(out, 0, a.shape, a), _out(out, 1, a.shape, a)
    sh = _stream_handle(stream, a.device)
    w = _workspace(linear_workspace_size(B, T, D), a.device, sh, ws)
    _check(load().mg_linear_scan_h0_fwd(a.data_ptr(), b.data_ptr(), _DT[a.dtype], h0.data_ptr(),
                                        A.data_ptr(), H.data_ptr(), B, T, D, w.data_ptr(),
                                        w.numel(), sh),
           "mg_linear_scan_h0_fwd")
    return A, H


def mg_linear_scan_h0_bwd(a, h0, A, H, gA, gH, *, out=None, ws=None, stream=None):
    """(da, db, dh0): gradients of sum(gA*A) + sum(gH*H) for mg_linear_scan_h0_fwd."""
    a = _prep(a, "a", (torch.float32, torch.bfloat16))
    h0, A, H, gA, gH = (_prep(x, n) for x, n in ((h0, "h0"), (A, "A"), (H, "H"), (gA, "gA"),
                                                  (gH, "gH")))
    if a.dim() != 3 or any(x.shape != a.shape for x in (A, H, gA, gH)) \
            or tuple(h0.shape) != (a.shape[0], a.shape[2]):
        raise ValueError("a, A, H, gA, gH must be (B, T, D) and h0 (B, D)")
    B, T, D = a.shape
    da, db = _out(out, 0, a.shape, a), _out(out, 1, a.shape, a)
    dh0 = _out(out, 2, h0.shape, a)
    sh = _stream_handle(stream, a.device)
    w = _workspace(linear_workspace_size(B, T, D), a.device, sh, ws)
    _check(load().mg_linear_scan_h0_bwd(a.data_ptr(), _DT[a.dtype], h0.data_ptr(), A.data_ptr(),
                                        H.data_ptr(), gA.data_ptr(), gH.data_ptr(), da.data_ptr(),
                                        db.data_ptr(), dh0.data_ptr(), B, T, D, w.data_ptr(),
                                        w.numel(), sh),
           "mg_linear_scan_h0_bwd")
    return da, db, dh0


def _cu(cu_seqlens, like):
    if not isinstance(cu_seqlens, torch.Tensor):
        cu_seqlens = torch.as_tensor(cu_seqlens, dtype=torch.int64)
    if cu_seqlens.dtype != torch.int64 or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens must be a 1-D int64 tensor of nseq + 1 offsets")
    return cu_seqlens.to(like.device).contiguous()


def mg_linear_scan_varlen_fwd(a, b, cu_seqlens, h0=None, *, out=None, ws=None, stream=None):
    """(A, H) float32 (Ttot, D) for packed sequences a, b (Ttot, D) with
    offsets cu_seqlens (nseq + 1, int64), each started from h0[s] ((nseq, D)
    float32) or 0."""
    a = _prep(a, "a", (torch.float32, torch.bfloat16))
    b = _prep(b, "b", (a.dtype,))
    cu = _cu(cu_seqlens, a)
    nseq = cu.numel() - 1
    if a.dim() != 2 or b.shape != a.shape:
        raise ValueError("a and b must both be (Ttot, D)")
    if h0 is not None:
        h0 = _prep(h0, "h0")
        if tuple(h0.shape) != (nseq, a.shape[1]):
            raise ValueError("h0 must be (nseq, D)")
    Ttot, D = a.shape
    A, H = _out(out, 0, a.shape, a), _out(out, 1, a.shape, a)
    sh = _stream_handle(stream, a.device)
    w = _workspace(varlen_workspace_size(Ttot, D), a.device, sh, ws)
    _check(load().mg_linear_scan_varlen_fwd(a.data_ptr(), b.data_ptr(), _DT[a.dtype],
                                            cu.data_ptr(), nseq,
                                            None if h0 is None else h0.data_ptr(), A.data_ptr(),
                                            H.data_ptr(), Ttot, D, w.data_ptr(), w.numel(), sh),
           "mg_linear_scan_varlen_fwd")
    return A, H


def mg_linear_scan_varlen_bwd(a, cu_seqlens, A, H, gA, gH, h0=None, *, out=None, ws=None,
                              stream=None):
    """(da, db, dh0) for mg_linear_scan_varlen_fwd; dh0 is None without h0."""
    a = _prep(a, "a", (torch.float32, torch.bfloat16))
    A, H, gA, gH = (_prep(x, n) for x, n in ((A, "A"), (H, "H"), (gA, "gA"), (gH, "gH")))
    cu = _cu(cu_seqlens, a)
    nseq = cu.numel() - 1
    if a.dim() != 2 or any(x.shape != a.shape for x in (A, H, gA, gH)):
        raise ValueError("a, A, H, gA, gH must all be (Ttot, D)")
    Ttot, D = a.shape
    dh0 = None
    if h0 is not None:
        h0 = _prep(h0, "h0")
        if tuple(h0.shape) != (nseq, D):
            raise ValueError("h0 must be (nseq, D)")
        dh0 = _out(out, 2, h0.shape, a)
    da, db = _out(out, 0, a.shape, a), _out(out, 1, a.shape, a)
    sh = _stream_handle(stream, a.device)
    w = _workspace(varlen_workspace_size(Ttot, D), a.device, sh, ws)
    ptr = lambda x: None if x is None else x.data_ptr()  # noqa: E731
    _check(load().mg_linear_scan_varlen_bwd(a.data_ptr(), _DT[a.dtype], cu.data_ptr(), nseq,
                                            ptr(h0), A.data_ptr(), H.data_ptr(), gA.data_ptr(),
                                            gH.data_ptr(), da.data_ptr(), db.data_ptr(), ptr(dh0),
                                            Ttot, D, w.data_ptr(), w.numel(), sh),
           "mg_linear_scan_varlen_bwd")
    return da, db, dh0


def mg_mingru_scan_fwd(x1, x2, *, want_A=True, out=None, ws=None, stream=None):
    """(A, Bc) float32 (B,T,D) of the linear scan on the minGRU gate
    a = 1 - sigmoid(x1), b = sigmoid(x1) g(x2), computed inside the scan.
    x1, x2: (B,T,D), both float32 or both bf16.  With want_A=False, A is not
    written and None is returned in its place."""
    x1 = _prep(x1, "x1", (torch.float32, torch.bfloat16))
    x2 = _prep(x2, "x2", (x1.dtype,))
    if x1.dim() != 3 or x2.shape != x1.shape:
        raise ValueError("x1 and x2 must both be (B, T, D)")
    B, T, D = x1.shape
    A = _out(out, 0, x1.shape, x1) if want_A else None
    Bc = _out(out, 1, x1.shape, x1)
    sh = _stream_handle(stream, x1.device)
    w = _workspace(mingru_workspace_size(B, T, D), x1.device, sh, ws)
    _check(load().mg_mingru_scan_fwd(x1.data_ptr(), x2.data_ptr(), _DT[x1.dtype],
                                     None if A is None else A.data_ptr(), Bc.data_ptr(), B, T, D,
                                     w.data_ptr(), w.numel(), sh),
           "mg_mingru_scan_fwd")
    return A, Bc


def mg_mingru_scan_bwd(x1, x2, A, Bc, gA, gBc, *, grad_dtype=torch.float32, out=None, ws=None,
                       stream=None):
    """(dx1, dx2) (B,T,D) of dtype grad_dtype: gradients of
    sum(gA*A) + sum(gBc*Bc) through the fused gate + scan.  A and gA may both
    be None (gA = 0, A not read)."""
    x1 = _prep(x1, "x1", (torch.float32, torch.bfloat16))
    x2 = _prep(x2, "x2", (x1.dtype,))
    if (A is None) != (gA is None):
        raise ValueError("A and gA must be given together (or both None)")
    Bc, gBc = _prep(Bc, "Bc"), _prep(gBc, "gBc")
    if A is not None:
        A, gA = _prep(A, "A"), _prep(gA, "gA")
    if x1.dim() != 3 or any(x is not None and x.shape != x1.shape for x in (x2, A, Bc, gA, gBc)):
        raise ValueError("x1, x2, A, Bc, gA, gBc must all be (B, T, D)")
    if grad_dtype not in _DT:
        raise ValueError("grad_dtype must be float32 or bfloat16")
    B, T, D = x1.shape
    dx1 = _out(out, 0, x1.shape, x1, grad_dtype)
    dx2 = _out(out, 1, x1.shape, x1, grad_dtype)
    sh = _stream_handle(stream, x1.device)
    w = _workspace(mingru_workspace_size(B, T, D), x1.device, sh, ws)
    ptr = lambda x: None if x is None else x.data_ptr()  # noqa: E731
    _check(load().mg_mingru_scan_bwd(x1.data_ptr(), x2.data_ptr(), _DT[x1.dtype], ptr(A),
                                     Bc.data_ptr(), ptr(gA), gBc.data_ptr(), dx1.data_ptr(),
                                     dx2.data_ptr(), _DT[grad_dtype], B, T, D, w.data_ptr(),
                                     w.numel(), sh),
           "mg_mingru_scan_bwd")
    return dx1, dx2


def mg_log_scan_fwd(log_coeffs, log_values, *, out=None, ws=None, stream=None):
    """h (B,T,D) float32 from log_coeffs (B,T,D) and log_values (B,T+1,D)."""
    lc = _prep(log_coeffs, "log_coeffs")
    lv = _prep(log_values, "log_values")
    if lc.dim() != 3:
        raise ValueError("log_coeffs must be (B, T, D)")
    B, T, D = lc.shape
    if tuple(lv.shape) != (B, T + 1, D):
        raise ValueError("log_values must be (B, T+1, D)")
    h = _out(None if out is None else (out,), 0, lc.shape, lc)
    sh = _stream_handle(stream, lc.device)
    w = _workspace(log_workspace_size(B, T, D), lc.device, sh, ws)
    _check(load().mg_log_scan_fwd(lc.data_ptr(), lv.data_ptr(), h.data_ptr(), B, T, D,
                                  w.data_ptr(), w.numel(), sh),
           "mg_log_scan_fwd")
    return h


def mg_log_scan_bwd(log_coeffs, log_values, h, gh, *, out=None, ws=None, stream=None):
    """(dlog_coeffs (B,T,D), dlog_values (B,T+1,D)) float32: gradients of
    sum(gh * h) for h = mg_log_scan_fwd(log_coeffs, log_values)."""
    lc = _prep(log_coeffs, "log_coeffs")
    lv = _prep(log_values, "log_values")
    h = _prep(h, "h")
    gh = _prep(gh, "gh")
    if lc.dim() != 3:
        raise ValueError("log_coeffs must be (B, T, D)")
    B, T, D = lc.shape
    if tuple(lv.shape) != (B, T + 1, D) or h.shape != lc.shape or gh.shape != lc.shape:
        raise ValueError("log_values must be (B, T+1, D); h and gh (B, T, D)")
    dlc = _out(out, 0, lc.shape, lc)
    dlv = _out(out, 1, lv.shape, lc)
    sh = _stream_handle(stream, lc.device)
    w = _workspace(log_workspace_size(B, T, D), lc.device, sh, ws)
    _check(load().mg_log_scan_bwd(lc.data_ptr(), lv.data_ptr(), h.data_ptr(), gh.data_ptr(),
                                  dlc.data_ptr(), dlv.data_ptr(), B, T, D, w.data_ptr(),
                                  w.numel(), sh),
           "mg_log_scan_bwd")
    return dlc, dlv


def mg_affine_scan_fwd(A, Bm, *, out=None, ws=None, stream=None):
    """(Abar, Bbar) for A (B,T,n,k,k), Bm (B,T,n,k,v), float32."""
    A = _prep(A, "A")
    Bm = _prep(Bm, "Bm")
    if A.dim() != 5 or A.shape[3] != A.shape[4] or Bm.dim() != 5 or Bm.shape[:4] != A.shape[:4]:
        raise ValueError("A must be (B,T,n,k,k) and Bm (B,T,n,k,v)")
    B, T, n, k, _ = A.shape
    v = Bm.shape[4]
    Abar, Bbar = _out(out, 0, A.shape, A), _out(out, 1, Bm.shape, A)
    sh = _stream_handle(stream, A.device)
    w = _workspace(affine_workspace_size(B, T, n, k, v), A.device, sh, ws)
    _check(load().mg_affine_scan_fwd(A.data_ptr(), Bm.data_ptr(), Abar.data_ptr(), Bbar.data_ptr(),
                                     B, T, n, k, v, w.data_ptr(), w.numel(), sh),
           "mg_affine_scan_fwd")
    return Abar, Bbar


def mg_affine_scan_bwd(A, Abar, Bbar, gAbar, gBbar, *, out=None, ws=None, stream=None):
    """(dA, dB): grads of <gAbar, Abar> + <gBbar, Bbar> w.r.t. A and Bm, float32."""
    A, Abar, Bbar, gAbar, gBbar = (_prep(x, nm) for x, nm in (
        (A, "A"), (Abar, "Abar"), (Bbar, "Bbar"), (gAbar, "gAbar"), (gBbar, "gBbar")))
    if A.dim() != 5 or Abar.shape != A.shape or gAbar.shape != A.shape \
            or Bbar.dim() != 5 or gBbar.shape != Bbar.shape or Bbar.shape[:4] != A.shape[:4]:
        raise ValueError("A, Abar, gAbar must be (B,T,n,k,k) and Bbar, gBbar (B,T,n,k,v)")
    B, T, n, k, _ = A.shape
    v = Bbar.shape[4]
    dA, dB = _out(out, 0, A.shape, A), _out(out, 1, Bbar.shape, A)
    sh = _stream_handle(stream, A.device)
    w = _workspace(affine_workspace_size(B, T, n, k, v), A.device, sh, ws)
    _check(load().mg_affine_scan_bwd(A.data_ptr(), Abar.data_ptr(), Bbar.data_ptr(),
                                     gAbar.data_ptr(), gBbar.data_ptr(), dA.data_ptr(),
                                     dB.data_ptr(), B, T, n, k, v, w.data_ptr(), w.numel(), sh),
           "mg_affine_scan_bwd")
    return dA, dB


def mg_affine_scan_h0_fwd(A, Bm, H0, *, out=None, ws=None, stream=None):
    """(Abar, Bbar) for A (B,T,n,k,k), Bm (B,T,n,k,v) started from H0 (B,n,k,v)."""
    A, Bm, H0 = _prep(A, "A"), _prep(Bm, "Bm"), _prep(H0, "H0")
    if A.dim() != 5 or A.shape[3] != A.shape[4] or Bm.dim() != 5 or Bm.shape[:4] != A.shape[:4]:
        raise ValueError("A must be (B,T,n,k,k) and Bm (B,T,n,k,v)")
    B, T, n, k, _ = A.shape
    v = Bm.shape[4]
    if tuple(H0.shape) != (B, n, k, v):
        raise ValueError("H0 must be (B, n, k, v)")
    Abar, Bbar = _out(out, 0, A.shape, A), _out(out, 1, Bm.shape, A)
    sh = _stream_handle(stream, A.device)
    w = _workspace(affine_workspace_size(B, T, n, k, v), A.device, sh, ws)
    _check(load().mg_affine_scan_h0_fwd(A.data_ptr(), Bm.data_ptr(), H0.data_ptr(),
                                        Abar.data_ptr(), Bbar.data_ptr(), B, T, n, k, v,
                                        w.data_ptr(), w.numel(), sh),
           "mg_affine_scan_h0_fwd")
    return Abar, Bbar


def mg_affine_scan_h0_bwd(A, H0, Abar, Bbar, gAbar, gBbar, *, out=None, ws=None, stream=None):
    """(dA, dB, dH0): gradients of <gAbar, Abar> + <gBbar, Bbar> for mg_affine_scan_h0_fwd."""
    A, H0, Abar, Bbar, gAbar, gBbar = (_prep(x, nm) for x, nm in (
        (A, "A"), (H0, "H0"), (Abar, "Abar"), (Bbar, "Bbar"), (gAbar, "gAbar"), (gBbar, "gBbar")))
    if A.dim() != 5 or Abar.shape != A.shape or gAbar.shape != A.shape \
            or Bbar.dim() != 5 or gBbar.shape != Bbar.shape or Bbar.shape[:4] != A.shape[:4]:
        raise ValueError("A, Abar, gAbar must be (B,T,n,k,k) and Bbar, gBbar (B,T,n,k,v)")
    B, T, n, k, _ = A.shape
    v = Bbar.shape[4]
    if tuple(H0.shape) != (B, n, k, v):
        raise ValueError("H0 must be (B, n, k, v)")
    dA, dB = _out(out, 0, A.shape, A), _out(out, 1, Bbar.shape, A)
    dH0 = _out(out, 2, H0.shape, A)
    sh = _stream_handle(stream, A.device)
    w = _workspace(affine_workspace_size(B, T, n, k, v), A.device, sh, ws)
    _check(load().mg_affine_scan_h0_bwd(A.data_ptr(), H0.data_ptr(), Abar.data_ptr(),
                                        Bbar.data_ptr(), gAbar.data_ptr(), gBbar.data_ptr(),
                                        dA.data_ptr(), dB.data_ptr(), dH0.data_ptr(), B, T, n, k,
                                        v, w.data_ptr(), w.numel(), sh),
           "mg_affine_scan_h0_bwd")
    return dA, dB, dH0


def _angle_consts(perm, sgn, p2p, R, k):
    """Host (R, k) arrays for the C ABI: perm, p2p int32, sgn float32 (p2p is
    the inverse of perm when not given)."""
    perm = torch.as_tensor(perm).detach().to("cpu", torch.int32).contiguous()
    sgn = torch.as_tensor(sgn).detach().to("cpu", torch.float32).contiguous()
    p2p = (torch.argsort(perm, dim=1) if p2p is None else torch.as_tensor(p2p)).detach() \
        .to("cpu", torch.int32).contiguous()
    if any(tuple(x.shape) != (R, k) for x in (perm, sgn, p2p)):
        raise ValueError("perm, sgn and p2p must be (R, k)")
    return perm, sgn, p2p


def mg_angle_scan_fwd(theta, scale, gamma, b, h0, perm, sgn, p2p=None, *, has_scale=1, has_decay=1,
                      out=None, stream=None):
    """h (B,T,n,k) of the angle-fused scan (Kernel 4); theta (B,T,n,R,k/2),
    scale, gamma (B,T,n), b (B,T,n,k), h0 (B,n,k) float32 on the device;
    perm, sgn, p2p (R,k) module constants (any device; copied to the host)."""
    theta, b, h0 = _prep(theta, "theta"), _prep(b, "b"), _prep(h0, "h0")
    if theta.dim() != 5 or b.dim() != 4:
        raise ValueError("theta must be (B,T,n,R,half) and b (B,T,n,k)")
    B, T, n, R, half = theta.shape
    k = 2 * half
    scale = _prep(scale, "scale") if has_scale else None
    gamma = _prep(gamma, "gamma") if has_decay else None
    if tuple(b.shape) != (B, T, n, k) or tuple(h0.shape) != (B, n, k) or any(
            x is not None and tuple(x.shape) != (B, T, n) for x in (scale, gamma)):
        raise ValueError("b must be (B,T,n,k), h0 (B,n,k), scale and gamma (B,T,n)")
    pm, sg, pp = _angle_consts(perm, sgn, p2p, R, k)
    h = _out(None if out is None else (out,), 0, b.shape, b)
    sh = _stream_handle(stream, b.device)
    ptr = lambda x: None if x is None else x.data_ptr()  # noqa: E731
    _check(load().mg_angle_scan_fwd(theta.data_ptr(), ptr(scale), ptr(gamma), b.data_ptr(),
                                    h0.data_ptr(), pm.data_ptr(), sg.data_ptr(), pp.data_ptr(),
                                    int(bool(has_scale)), int(bool(has_decay)), h.data_ptr(), B, T,
                                    n, R, k, sh),
           "mg_angle_scan_fwd")
    return h


def mg_angle_scan_bwd(theta, scale, gamma, h0, out_h, grad_out, perm, sgn, p2p=None, *,
                      has_scale=1, has_decay=1, out=None, stream=None):
    """(dtheta, dscale, dgamma, db, dh0) of sum(grad_out * h) for the angle
    scan, from the stored states out_h = h."""
    theta, h0 = _prep(theta, "theta"), _prep(h0, "h0")
    out_h, grad_out = _prep(out_h, "out"), _prep(grad_out, "grad_out")
    B, T, n, R, half = theta.shape
    k = 2 * half
    scale = _prep(scale, "scale") if has_scale else None
    gamma = _prep(gamma, "gamma") if has_decay else None
    if tuple(out_h.shape) != (B, T, n, k) or grad_out.shape != out_h.shape \
            or tuple(h0.shape) != (B, n, k):
        raise ValueError("out, grad_out must be (B,T,n,k) and h0 (B,n,k)")
    pm, sg, pp = _angle_consts(perm, sgn, p2p, R, k)
    dth = _out(out, 0, theta.shape, theta)
    dsc = _out(out, 1, (B, T, n), theta)
    dga = _out(out, 2, (B, T, n), theta)
    db = _out(out, 3, out_h.shape, theta)
    dh0 = _out(out, 4, h0.shape, theta)
    sh = _stream_handle(stream, theta.device)
    ptr = lambda x: None if x is None else x.data_ptr()  # noqa: E731
    _check(load().mg_angle_scan_bwd(theta.data_ptr(), ptr(scale), ptr(gamma), h0.data_ptr(),
                                    out_h.data_ptr(), grad_out.data_ptr(), pm.data_ptr(),
                                    sg.data_ptr(), pp.data_ptr(), int(bool(has_scale)),
                                    int(bool(has_decay)), dth.data_ptr(), dsc.data_ptr(),
                                    dga.data_ptr(), db.data_ptr(), dh0.data_ptr(), B, T, n, R, k,
                                    sh),
           "mg_angle_scan_bwd")
    return dth, dsc, dga, db, dh0


def mg_linear_scan_fwd_noalloc(a, b, *, out=None, stream=None):
    """mg_linear_scan_fwd with the library's static scratch instead of a
    workspace: the C entry point allocates nothing (for callers that cannot
    allocate device memory at call time).  Outputs are allocated here unless
    given; calls that overlap on the GPU must be serialised by the caller."""
    a = _prep(a, "a", (torch.float32, torch.bfloat16))
    b = _prep(b, "b", (a.dtype,))
    if a.dim() != 3 or b.shape != a.shape:
        raise ValueError("a and b must both be (B, T, D)")
    B, T, D = a.shape
    A, Bc = _out(out, 0, a.shape, a), _out(out, 1, a.shape, a)
    sh = _stream_handle(stream, a.device)
    _check(load().mg_linear_scan_fwd_noalloc(a.data_ptr(), b.data_ptr(), _DT[a.dtype],
                                             A.data_ptr(), Bc.data_ptr(), B, T, D, sh),
           "mg_linear_scan_fwd_noalloc")
    return A, Bc


def noalloc_status(stream=None, device=None) -> None:
    """Raise MgScanError if a device-side wait of a mg_linear_scan_fwd_noalloc
    call on the current device gave up since the last check (synchronises
    the stream)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _check(load().mg_linear_scan_fwd_noalloc_status(_stream_handle(stream, dev)),
           "mg_linear_scan_fwd_noalloc_status")


# Names of the page "minGRU - Triton kernels".
linear_scan_fwd = mg_linear_scan_fwd
linear_scan_bwd = mg_linear_scan_bwd
parallel_scan_log_fwd = mg_log_scan_fwd
parallel_scan_log_bwd = mg_log_scan_bwd
affine_scan_fwd = mg_affine_scan_fwd
affine_scan_bwd = mg_affine_scan_bwd
mingru_scan_fwd = mg_mingru_scan_fwd
mingru_scan_bwd = mg_mingru_scan_bwd
linear_scan_h0_fwd = mg_linear_scan_h0_fwd
linear_scan_h0_bwd = mg_linear_scan_h0_bwd
linear_scan_varlen_fwd = mg_linear_scan_varlen_fwd
linear_scan_varlen_bwd = mg_linear_scan_varlen_bwd
affine_scan_h0_fwd = mg_affine_scan_h0_fwd
affine_scan_h0_bwd = mg_affine_scan_h0_bwd
angle_scan_fwd = mg_angle_scan_fwd
angle_scan_bwd = mg_angle_scan_bwd
