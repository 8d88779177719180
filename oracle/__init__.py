"""Float64 CPU oracle for the minGRU scan family.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never imports it and
shares no code with it.

Each function is the plain sequential definition of one op of the
``mingru.triton_scans`` API reference page (page "minGRU - Triton kernels"),
evaluated in double precision by ``mg_oracle.c``:

* ``linear_scan_fwd``   -- linear_scan_fwd: running product A, h_0 = 0 solution Bc
* ``linear_scan_bwd``   -- linear_scan_bwd: da, db from a, A, Bc, gA, gBc
* ``log_scan_fwd``      -- parallel_scan_log_fwd: h_1..h_T from log_coeffs, log_values
* ``affine_scan_fwd``   -- affine_scan_fwd: Abar (running matrix product), Bbar
* ``affine_scan_bwd``   -- affine_scan_bwd: dA, dB
* ``mingru_gate``, ``mingru_scan_fwd``, ``mingru_scan_bwd`` -- the minGRU gate
  (a = 1 - sigmoid(x1), b = sigmoid(x1) g(x2)) fused with the linear scan, and
  its gradients with respect to x1, x2
* ``linear_scan_varlen_fwd/bwd``, ``linear_scan_h0_fwd/bwd`` -- the linear
  scan from a start state h0, over (B,T,D) or a packed variable-length batch
* ``affine_scan_h0_fwd/bwd`` -- the affine scan from a start state H0
* ``angle_scan_fwd/bwd`` -- the angle-fused scan (Kernel 4) under the reading
  stated in mg_oracle.c (parity of that reading is unpinned by the page)

Inputs are converted to contiguous float64 numpy arrays (a float32 or bf16
value widens exactly).  Outputs are float64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mg_oracle.c")
_LIB = os.path.join(_HERE, "libmgoracle.so")


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile ``src`` (default ``mg_oracle.c``) into the shared library ``out``
    (gcc, -O2, no fast-math, no FMA contraction).  Returns the library path."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
           "-shared", "-fPIC", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _f64(x) -> np.ndarray:
    """Contiguous float64 copy of a numpy array or a torch tensor (bf16 widens exactly)."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu", torch.float64).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x: np.ndarray):
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


class Oracle:
    """The oracle functions bound to one build of the C source."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P = ctypes.POINTER(ctypes.c_double)
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.orc_linear_scan_fwd.argtypes = [P, P, P, P, I64, I64, I64]
        lib.orc_linear_scan_bwd.argtypes = [P, P, P, P, P, P, P, I64, I64, I64]
        lib.orc_log_scan_fwd.argtypes = [P, P, P, I64, I64, I64]
        lib.orc_log_scan_bwd.argtypes = [P, P, P, P, P, I64, I64, I64]
        lib.orc_affine_scan_fwd.argtypes = [P, P, P, P, I64, I64, I64, I, I]
        lib.orc_affine_scan_bwd.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I, I]
        PI = ctypes.POINTER(ctypes.c_int64)
        lib.orc_mingru_gate.argtypes = [P, P, P, P, I64]
        lib.orc_mingru_scan_fwd.argtypes = [P, P, P, P, I64, I64, I64]
        lib.orc_mingru_scan_bwd.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64]
        lib.orc_linear_scan_varlen_fwd.argtypes = [P, P, PI, I64, P, P, P, I64]
        lib.orc_linear_scan_varlen_bwd.argtypes = [P, PI, I64, P, P, P, P, P, P, P, P, I64]
        lib.orc_affine_scan_h0_fwd.argtypes = [P, P, P, P, P, I64, I64, I64, I, I]
        lib.orc_affine_scan_h0_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I64, I64, I64, I, I]
        PI32 = ctypes.POINTER(ctypes.c_int32)
        lib.orc_angle_scan_fwd.argtypes = [P, P, P, P, P, PI32, P, I, I, P, I64, I64, I64, I, I]
        lib.orc_angle_scan_bwd.argtypes = [P, P, P, P, P, P, PI32, P, I, I, P, P, P, P, P, I64, I64,
                                           I64, I, I]
        lib.orc_angle_scan_fwd.restype = None
        lib.orc_angle_scan_bwd.restype = None
        for f in (lib.orc_linear_scan_fwd, lib.orc_linear_scan_bwd, lib.orc_log_scan_fwd,
                  lib.orc_log_scan_bwd, lib.orc_affine_scan_fwd, lib.orc_affine_scan_bwd,
                  lib.orc_mingru_gate, lib.orc_mingru_scan_fwd, lib.orc_mingru_scan_bwd,
                  lib.orc_linear_scan_varlen_fwd, lib.orc_linear_scan_varlen_bwd,
                  lib.orc_affine_scan_h0_fwd, lib.orc_affine_scan_h0_bwd):
            f.restype = None
        self._lib = lib

    def linear_scan_fwd(self, a, b):
        """(A, Bc) for a, b (B,T,D): A_t = a_t A_{t-1}, Bc_t = a_t Bc_{t-1} + b_t."""
        a, b = _f64(a), _f64(b)
        assert a.ndim == 3 and a.shape == b.shape
        A = np.empty_like(a)
        Bc = np.empty_like(a)
        self._lib.orc_linear_scan_fwd(_ptr(a), _ptr(b), _ptr(A), _ptr(Bc), *a.shape)
        return A, Bc

    def linear_scan_bwd(self, a, A, Bc, gA, gBc):
        """(da, db) for L = sum(gA*A) + sum(gBc*Bc), with A, Bc taken as given."""
        a, A, Bc, gA, gBc = (_f64(x) for x in (a, A, Bc, gA, gBc))
        assert a.ndim == 3 and all(x.shape == a.shape for x in (A, Bc, gA, gBc))
        da = np.empty_like(a)
        db = np.empty_like(a)
        self._lib.orc_linear_scan_bwd(_ptr(a), _ptr(A), _ptr(Bc), _ptr(gA), _ptr(gBc),
                                      _ptr(da), _ptr(db), *a.shape)
        return da, db

    def log_scan_fwd(self, log_coeffs, log_values):
        """h_1..h_T (B,T,D) for log_coeffs (B,T,D), log_values (B,T+1,D)."""
        lc, lv = _f64(log_coeffs), _f64(log_values)
        B, T, D = lc.shape
        assert lv.shape == (B, T + 1, D)
        h = np.empty_like(lc)
        self._lib.orc_log_scan_fwd(_ptr(lc), _ptr(lv), _ptr(h), B, T, D)
        return h

    def log_scan_bwd(self, log_coeffs, log_values, gh):
        """(dlog_coeffs (B,T,D), dlog_values (B,T+1,D)) for L = sum(gh * h)."""
        lc, lv, g = _f64(log_coeffs), _f64(log_values), _f64(gh)
        B, T, D = lc.shape
        assert lv.shape == (B, T + 1, D) and g.shape == lc.shape
        dlc = np.empty_like(lc)
        dlv = np.empty_like(lv)
        self._lib.orc_log_scan_bwd(_ptr(lc), _ptr(lv), _ptr(g), _ptr(dlc), _ptr(dlv), B, T, D)
        return dlc, dlv

    def affine_scan_fwd(self, A, Bm):
        """(Abar, Bbar) for A (B,T,n,k,k), Bm (B,T,n,k,v)."""
        A, Bm = _f64(A), _f64(Bm)
        B, T, n, k, k2 = A.shape
        assert k == k2 and Bm.shape[:4] == (B, T, n, k)
        v = Bm.shape[4]
        Abar = np.empty_like(A)
        Bbar = np.empty_like(Bm)
        self._lib.orc_affine_scan_fwd(_ptr(A), _ptr(Bm), _ptr(Abar), _ptr(Bbar),
                                      B, T, n, k, v)
        return Abar, Bbar

    def affine_scan_bwd(self, A, Abar, Bbar, gAbar, gBbar):
        """(dA, dB) for L = <gAbar, Abar> + <gBbar, Bbar>, with Abar, Bbar taken as given."""
        A, Abar, Bbar, gAbar, gBbar = (_f64(x) for x in (A, Abar, Bbar, gAbar, gBbar))
        B, T, n, k, _ = A.shape
        v = Bbar.shape[4]
        assert Abar.shape == A.shape and gAbar.shape == A.shape
        assert Bbar.shape == (B, T, n, k, v) and gBbar.shape == Bbar.shape
        dA = np.empty_like(A)
        dB = np.empty_like(Bbar)
        self._lib.orc_affine_scan_bwd(_ptr(A), _ptr(Abar), _ptr(Bbar), _ptr(gAbar),
                                      _ptr(gBbar), _ptr(dA), _ptr(dB), B, T, n, k, v)
        return dA, dB


    # -------------------------------------------- fused minGRU gate + scan

    def mingru_gate(self, x1, x2):
        """(a, b) = (1 - sigmoid(x1), sigmoid(x1) g(x2)), elementwise."""
        x1, x2 = _f64(x1), _f64(x2)
        assert x1.shape == x2.shape
        a, b = np.empty_like(x1), np.empty_like(x1)
        self._lib.orc_mingru_gate(_ptr(x1), _ptr(x2), _ptr(a), _ptr(b), x1.size)
        return a, b

    def mingru_scan_fwd(self, x1, x2):
        """(A, Bc) of the linear scan on the minGRU gate of x1, x2 (B,T,D)."""
        x1, x2 = _f64(x1), _f64(x2)
        assert x1.ndim == 3 and x1.shape == x2.shape
        A, Bc = np.empty_like(x1), np.empty_like(x1)
        self._lib.orc_mingru_scan_fwd(_ptr(x1), _ptr(x2), _ptr(A), _ptr(Bc), *x1.shape)
        return A, Bc

    def mingru_scan_bwd(self, x1, x2, A, Bc, gA, gBc):
        """(dx1, dx2) for L = sum(gA*A) + sum(gBc*Bc), A and Bc taken as given."""
        x1, x2, A, Bc, gA, gBc = (_f64(x) for x in (x1, x2, A, Bc, gA, gBc))
        assert x1.ndim == 3 and all(x.shape == x1.shape for x in (x2, A, Bc, gA, gBc))
        dx1, dx2 = np.empty_like(x1), np.empty_like(x1)
        self._lib.orc_mingru_scan_bwd(_ptr(x1), _ptr(x2), _ptr(A), _ptr(Bc), _ptr(gA), _ptr(gBc),
                                      _ptr(dx1), _ptr(dx2), *x1.shape)
        return dx1, dx2

    # ------------------------------------------ start states, varlen batches

    @staticmethod
    def _cu(cu, Ttot):
        cu = np.ascontiguousarray(np.asarray(cu, dtype=np.int64))
        assert cu.ndim == 1 and cu[0] == 0 and cu[-1] == Ttot and np.all(np.diff(cu) >= 0)
        return cu

    def linear_scan_varlen_fwd(self, a, b, cu_seqlens, h0=None):
        """(A, H) over packed rows a, b (Ttot, D); sequence s is rows
        cu[s]..cu[s+1]-1, started from h0[s] (nseq, D) or 0."""
        a, b = _f64(a), _f64(b)
        assert a.ndim == 2 and a.shape == b.shape
        cu = self._cu(cu_seqlens, a.shape[0])
        nseq = cu.size - 1
        h = None if h0 is None else _f64(h0)
        assert h is None or h.shape == (nseq, a.shape[1])
        A, H = np.empty_like(a), np.empty_like(a)
        self._lib.orc_linear_scan_varlen_fwd(_ptr(a), _ptr(b), cu.ctypes.data_as(
            ctypes.POINTER(ctypes.c_int64)), nseq, None if h is None else _ptr(h), _ptr(A), _ptr(H),
            a.shape[1])
        return A, H

    def linear_scan_varlen_bwd(self, a, cu_seqlens, A, H, gA, gH, h0=None):
        """(da, db, dh0) for L = sum(gA*A) + sum(gH*H); dh0 is None without h0."""
        a, A, H, gA, gH = (_f64(x) for x in (a, A, H, gA, gH))
        assert a.ndim == 2 and all(x.shape == a.shape for x in (A, H, gA, gH))
        cu = self._cu(cu_seqlens, a.shape[0])
        nseq = cu.size - 1
        h = None if h0 is None else _f64(h0)
        da, db = np.empty_like(a), np.empty_like(a)
        dh0 = None if h is None else np.empty_like(h)
        self._lib.orc_linear_scan_varlen_bwd(
            _ptr(a), cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), nseq,
            None if h is None else _ptr(h), _ptr(A), _ptr(H), _ptr(gA), _ptr(gH), _ptr(da), _ptr(db),
            None if dh0 is None else _ptr(dh0), a.shape[1])
        return da, db, dh0

    def linear_scan_h0_fwd(self, a, b, h0):
        """(A, H) for a, b (B,T,D) with start states h0 (B,D): the varlen op on
        B sequences of length T."""
        a, b = _f64(a), _f64(b)
        Bn, T, D = a.shape
        A, H = self.linear_scan_varlen_fwd(a.reshape(Bn * T, D), b.reshape(Bn * T, D),
                                           np.arange(Bn + 1) * T, h0)
        return A.reshape(a.shape), H.reshape(a.shape)

    def linear_scan_h0_bwd(self, a, h0, A, H, gA, gH):
        """(da, db, dh0) for the (B,T,D) forward with start states h0 (B,D)."""
        a = _f64(a)
        Bn, T, D = a.shape
        flat = lambda x: _f64(x).reshape(Bn * T, D)  # noqa: E731
        da, db, dh0 = self.linear_scan_varlen_bwd(flat(a), np.arange(Bn + 1) * T, flat(A), flat(H),
                                                  flat(gA), flat(gH), h0)
        return da.reshape(a.shape), db.reshape(a.shape), dh0

    def affine_scan_h0_fwd(self, A, Bm, H0):
        """(Abar, Bbar) for A (B,T,n,k,k), Bm (B,T,n,k,v) started from H0 (B,n,k,v)."""
        A, Bm, H0 = _f64(A), _f64(Bm), _f64(H0)
        B, T, n, k, _ = A.shape
        v = Bm.shape[4]
        assert H0.shape == (B, n, k, v)
        Abar, Bbar = np.empty_like(A), np.empty_like(Bm)
        self._lib.orc_affine_scan_h0_fwd(_ptr(A), _ptr(Bm), _ptr(H0), _ptr(Abar), _ptr(Bbar),
                                         B, T, n, k, v)
        return Abar, Bbar

    def affine_scan_h0_bwd(self, A, H0, Abar, Bbar, gAbar, gBbar):
        """(dA, dB, dH0) for L = <gAbar, Abar> + <gBbar, Bbar> with start state H0."""
        A, H0, Abar, Bbar, gAbar, gBbar = (_f64(x) for x in (A, H0, Abar, Bbar, gAbar, gBbar))
        B, T, n, k, _ = A.shape
        v = Bbar.shape[4]
        dA, dB, dH0 = np.empty_like(A), np.empty_like(Bbar), np.empty_like(H0)
        self._lib.orc_affine_scan_h0_bwd(_ptr(A), _ptr(H0), _ptr(Abar), _ptr(Bbar), _ptr(gAbar),
                                         _ptr(gBbar), _ptr(dA), _ptr(dB), _ptr(dH0), B, T, n, k, v)
        return dA, dB, dH0

    # ---------------------------------------------------- angle-fused scan

    @staticmethod
    def _perm(perm, R, k):
        perm = np.ascontiguousarray(np.asarray(perm, dtype=np.int32))
        assert perm.shape == (R, k) and all(sorted(r) == list(range(k)) for r in perm.tolist())
        return perm

    def angle_scan_fwd(self, theta, scale, gamma, b, h0, perm, sgn, has_scale=1, has_decay=1):
        """h (B,T,n,k) of the angle-fused scan (reading in mg_oracle.c)."""
        theta, scale, gamma, b, h0, sgn = (_f64(x) for x in (theta, scale, gamma, b, h0, sgn))
        B, T, n, R, half = theta.shape
        k = 2 * half
        assert scale.shape == (B, T, n) and gamma.shape == (B, T, n)
        assert b.shape == (B, T, n, k) and h0.shape == (B, n, k) and sgn.shape == (R, k)
        perm = self._perm(perm, R, k)
        h = np.empty_like(b)
        self._lib.orc_angle_scan_fwd(_ptr(theta), _ptr(scale), _ptr(gamma), _ptr(b), _ptr(h0),
                                     perm.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), _ptr(sgn),
                                     int(has_scale), int(has_decay), _ptr(h), B, T, n, R, k)
        return h

    def angle_scan_bwd(self, theta, scale, gamma, h0, out, grad_out, perm, sgn, has_scale=1,
                       has_decay=1):
        """(dtheta, dscale, dgamma, db, dh0) for L = sum(grad_out * h), out = h as given."""
        theta, scale, gamma, h0, out, grad_out, sgn = (
            _f64(x) for x in (theta, scale, gamma, h0, out, grad_out, sgn))
        B, T, n, R, half = theta.shape
        k = 2 * half
        assert out.shape == (B, T, n, k) and grad_out.shape == out.shape
        perm = self._perm(perm, R, k)
        dtheta, dscale, dgamma = np.empty_like(theta), np.empty_like(scale), np.empty_like(gamma)
        db, dh0 = np.empty_like(out), np.empty_like(h0)
        self._lib.orc_angle_scan_bwd(_ptr(theta), _ptr(scale), _ptr(gamma), _ptr(h0), _ptr(out),
                                     _ptr(grad_out),
                                     perm.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), _ptr(sgn),
                                     int(has_scale), int(has_decay), _ptr(dtheta), _ptr(dscale),
                                     _ptr(dgamma), _ptr(db), _ptr(dh0), B, T, n, R, k)
        return dtheta, dscale, dgamma, db, dh0


_default = None


def _oracle() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def linear_scan_fwd(a, b):
    return _oracle().linear_scan_fwd(a, b)


def linear_scan_bwd(a, A, Bc, gA, gBc):
    return _oracle().linear_scan_bwd(a, A, Bc, gA, gBc)


def log_scan_fwd(log_coeffs, log_values):
    return _oracle().log_scan_fwd(log_coeffs, log_values)


def log_scan_bwd(log_coeffs, log_values, gh):
    return _oracle().log_scan_bwd(log_coeffs, log_values, gh)


def affine_scan_fwd(A, Bm):
    return _oracle().affine_scan_fwd(A, Bm)


def affine_scan_bwd(A, Abar, Bbar, gAbar, gBbar):
    return _oracle().affine_scan_bwd(A, Abar, Bbar, gAbar, gBbar)


def mingru_gate(x1, x2):
    return _oracle().mingru_gate(x1, x2)


def mingru_scan_fwd(x1, x2):
    return _oracle().mingru_scan_fwd(x1, x2)


def mingru_scan_bwd(x1, x2, A, Bc, gA, gBc):
    return _oracle().mingru_scan_bwd(x1, x2, A, Bc, gA, gBc)


def linear_scan_varlen_fwd(a, b, cu_seqlens, h0=None):
    return _oracle().linear_scan_varlen_fwd(a, b, cu_seqlens, h0)


def linear_scan_varlen_bwd(a, cu_seqlens, A, H, gA, gH, h0=None):
    return _oracle().linear_scan_varlen_bwd(a, cu_seqlens, A, H, gA, gH, h0)


def linear_scan_h0_fwd(a, b, h0):
    return _oracle().linear_scan_h0_fwd(a, b, h0)


def linear_scan_h0_bwd(a, h0, A, H, gA, gH):
    return _oracle().linear_scan_h0_bwd(a, h0, A, H, gA, gH)


def affine_scan_h0_fwd(A, Bm, H0):
    return _oracle().affine_scan_h0_fwd(A, Bm, H0)


def affine_scan_h0_bwd(A, H0, Abar, Bbar, gAbar, gBbar):
    return _oracle().affine_scan_h0_bwd(A, H0, Abar, Bbar, gAbar, gBbar)


def angle_scan_fwd(theta, scale, gamma, b, h0, perm, sgn, has_scale=1, has_decay=1):
    return _oracle().angle_scan_fwd(theta, scale, gamma, b, h0, perm, sgn, has_scale, has_decay)


def angle_scan_bwd(theta, scale, gamma, h0, out, grad_out, perm, sgn, has_scale=1, has_decay=1):
    return _oracle().angle_scan_bwd(theta, scale, gamma, h0, out, grad_out, perm, sgn, has_scale,
                                    has_decay)
