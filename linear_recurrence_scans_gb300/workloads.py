"""Seeded synthetic inputs for the minGRU scan family.

This module draws random numbers and shapes them into the workloads the scan
ops are measured and checked on.  It holds none of the scans' arithmetic, so
both the CUDA path (bench, GPU tests) and the float64 oracle (tests) can take
their inputs from it without sharing any of the method.

Each tensor gets its own seeded torch generator: sub-stream ``seed + i`` for
the i-th tensor in the order listed in each function's docstring.  Every
tensor is returned as float32 unless stated otherwise; bf16 variants are the
float32 draw rounded to bf16.

Workloads (the minGRU reading of the scan ops on the page "minGRU - Triton
kernels"):

* ``uniform_linear``   a ~ U(0,1), b ~ N(0,1)                       (B,T,D)
* ``mingru_linear``    x1,x2 ~ N(0,1); z = sigmoid(x1); a = 1 - z;
                       b = z * g(x2), g(x) = x + 0.5 (x >= 0) else sigmoid(x);
                       gA, gBc ~ N(0,1)                              (B,T,D)
* ``mingru_x``         x1, x2 ~ N(0,1) raw (the fused gate + scan's inputs);
                       gA, gBc ~ N(0,1)
* ``mingru_log``       k, x ~ N(0,1); log_coeffs = -softplus(k);
                       log_values[:, 0] = log 0.5,
                       log_values[:, t] = -softplus(-k_{t-1}) + log g(x_{t-1})
* ``angle_inputs``     theta ~ U(-pi, pi), scale = tanh(N(0,1)), gamma =
                       exp(-U(0, 0.3)), b, h0 ~ N(0,1), seeded perm/sgn
* ``haar_affine``      A_t = 0.95 * Q_t, Q_t Haar on O(k) (QR of a float64
                       N(0,1) matrix with the sign fix Q diag(sign diag R));
                       Bm, gAbar, gBbar ~ N(0,1)
"""
from __future__ import annotations

import math

import torch


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def g_act(x: torch.Tensor) -> torch.Tensor:
    """minGRU's positive activation: x + 0.5 for x >= 0, sigmoid(x) otherwise."""
    return torch.where(x >= 0, x + 0.5, torch.sigmoid(x))


def uniform_linear(B: int, T: int, D: int, seed: int = 0, device="cpu"):
    """(a, b): a ~ U(0,1) (stream seed), b ~ N(0,1) (stream seed+1)."""
    a = torch.rand((B, T, D), generator=_gen(seed, device), device=device, dtype=torch.float32)
    b = torch.randn((B, T, D), generator=_gen(seed + 1, device), device=device, dtype=torch.float32)
    return a, b


def mingru_linear(B: int, T: int, D: int, seed: int = 0, device="cpu",
                  in_dtype=torch.float32, grads: bool = True):
    """(a, b, gA, gBc) shaped like a minGRU layer's scan.

    Streams: x1 (seed), x2 (seed+1), gA (seed+2), gBc (seed+3).  a and b are
    computed in float32 and then cast to ``in_dtype``; gA, gBc are float32.
    """
    shape = (B, T, D)
    x1 = torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    z = torch.sigmoid(x1)
    del x1
    a = (1.0 - z).to(in_dtype)
    x2 = torch.randn(shape, generator=_gen(seed + 1, device), device=device, dtype=torch.float32)
    b = (z * g_act(x2)).to(in_dtype)
    del x2, z
    if not grads:
        return a, b, None, None
    gA = torch.randn(shape, generator=_gen(seed + 2, device), device=device, dtype=torch.float32)
    gBc = torch.randn(shape, generator=_gen(seed + 3, device), device=device, dtype=torch.float32)
    return a, b, gA, gBc


def mingru_x(B: int, T: int, D: int, seed: int = 0, device="cpu", in_dtype=torch.float32,
             grads: bool = True):
    """(x1, x2, gA, gBc): the two gate projections of a minGRU layer, drawn
    as in ``mingru_linear`` (same streams and seeds, so the gate of these x1,
    x2 is that workload's a, b) but returned raw, for the fused gate + scan.
    x1, x2 are cast to ``in_dtype``; gA, gBc are float32."""
    shape = (B, T, D)
    x1 = torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    x2 = torch.randn(shape, generator=_gen(seed + 1, device), device=device, dtype=torch.float32)
    x1, x2 = x1.to(in_dtype), x2.to(in_dtype)
    if not grads:
        return x1, x2, None, None
    gA = torch.randn(shape, generator=_gen(seed + 2, device), device=device, dtype=torch.float32)
    gBc = torch.randn(shape, generator=_gen(seed + 3, device), device=device, dtype=torch.float32)
    return x1, x2, gA, gBc


def mingru_log(B: int, T: int, D: int, seed: int = 0, device="cpu"):
    """(log_coeffs (B,T,D), log_values (B,T+1,D)).  Streams: k (seed), x (seed+1).

    The same draw k_t feeds log_coeffs[:, t] and log_values[:, t+1], as in a
    minGRU layer where log(1 - z_t) and log(z_t) come from one gate logit.
    """
    k = torch.randn((B, T, D), generator=_gen(seed, device), device=device, dtype=torch.float32)
    x = torch.randn((B, T, D), generator=_gen(seed + 1, device), device=device, dtype=torch.float32)
    log_coeffs = -torch.nn.functional.softplus(k)
    log_values = torch.empty((B, T + 1, D), device=device, dtype=torch.float32)
    log_values[:, 0] = math.log(0.5)
    log_values[:, 1:] = -torch.nn.functional.softplus(-k) + torch.log(g_act(x))
    return log_coeffs, log_values


def haar_orthogonal(count: int, k: int, seed: int) -> torch.Tensor:
    """``count`` independent Haar-random k x k orthogonal matrices, float64 (CPU)."""
    z = torch.randn((count, k, k), generator=_gen(seed), dtype=torch.float64)
    q, r = torch.linalg.qr(z)
    d = torch.diagonal(r, dim1=-2, dim2=-1)
    s = torch.where(d < 0, -torch.ones_like(d), torch.ones_like(d))
    return q * s.unsqueeze(-2)


def haar_affine(B: int, T: int, n: int, k: int, v: int, seed: int = 0, device="cpu",
                grads: bool = True, decay: float = 0.95):
    """(A, Bm, gAbar, gBbar): A (B,T,n,k,k) = decay * Haar, the rest N(0,1).

    Streams: Q (seed), Bm (seed+1), gAbar (seed+2), gBbar (seed+3).  The Haar
    draw is made on the CPU in float64 and rounded to float32 after scaling.
    """
    q = haar_orthogonal(B * T * n, k, seed)
    A = (decay * q).to(torch.float32).reshape(B, T, n, k, k).contiguous().to(device)
    Bm = torch.randn((B, T, n, k, v), generator=_gen(seed + 1), dtype=torch.float32).to(device)
    if not grads:
        return A, Bm, None, None
    gAbar = torch.randn((B, T, n, k, k), generator=_gen(seed + 2), dtype=torch.float32).to(device)
    gBbar = torch.randn((B, T, n, k, v), generator=_gen(seed + 3), dtype=torch.float32).to(device)
    return A, Bm, gAbar, gBbar


def angle_inputs(B: int, T: int, n: int, R: int, k: int, seed: int = 0, device="cpu",
                 grads: bool = True):
    """Inputs of the angle-fused scan: theta (B,T,n,R,k/2) ~ U(-pi, pi);
    scale = tanh(u), u ~ N(0,1) and gamma = exp(-lambda), lambda ~ U(0, 0.3)
    (the module's parameterisations), both (B,T,n); b (B,T,n,k), h0 (B,n,k)
    ~ N(0,1); perm (R,k) int32, one seeded permutation per layer, p2p its
    inverse, sgn (R,k) float32 in {-1, +1} (CPU arrays, module constants);
    grad_out (B,T,n,k) ~ N(0,1).  Streams seed .. seed+6 in that order."""
    th = (torch.rand((B, T, n, R, k // 2), generator=_gen(seed, device), device=device) * 2 - 1) * math.pi
    scale = torch.tanh(torch.randn((B, T, n), generator=_gen(seed + 1, device), device=device))
    gamma = torch.exp(-0.3 * torch.rand((B, T, n), generator=_gen(seed + 2, device), device=device))
    b = torch.randn((B, T, n, k), generator=_gen(seed + 3, device), device=device)
    h0 = torch.randn((B, n, k), generator=_gen(seed + 4, device), device=device)
    g = _gen(seed + 5)
    perm = torch.stack([torch.randperm(k, generator=g) for _ in range(R)]).to(torch.int32)
    p2p = torch.argsort(perm, dim=1).to(torch.int32)
    sgn = torch.where(torch.rand((R, k), generator=g) < 0.5, -1.0, 1.0).to(torch.float32)
    go = torch.randn((B, T, n, k), generator=_gen(seed + 6, device), device=device) if grads else None
    return th, scale, gamma, b, h0, perm, sgn, p2p, go


# The workloads the library is checked and measured on, by name.
CONFIGS = {
    # linear_scan_fwd fp32, a ~ U(0,1), b ~ N(0,1)
    "uniform_linear_2x256x64": dict(op="linear", B=2, T=256, D=64),
    # minGRU-shaped linear_scan fwd+bwd fp32
    "mingru_linear_8x4096x1024": dict(op="linear", B=8, T=4096, D=1024),
    # parallel_scan_log_fwd fp32
    "mingru_log_16x2048x2048": dict(op="log", B=16, T=2048, D=2048),
    # affine_scan fwd+bwd fp32, Haar-decayed 4x4 and 16x16 transitions
    "haar_affine_4x2048x64_k4v4": dict(op="affine", B=4, T=2048, n=64, k=4, v=4),
    "haar_affine_2x1024x32_k16v16": dict(op="affine", B=2, T=1024, n=32, k=16, v=16),
    # large minGRU linear_scan fwd+bwd with bf16 a, b; fp32 accumulation and outputs
    "mingru_linear_bf16_16x32768x4096": dict(op="linear", B=16, T=32768, D=4096, bf16=True),
}
