"""Run one op of the library on one named workload a few times (for profilers).

    python -m linear_recurrence_scans_gb300.run_case <case> [repeats]

Cases (inputs seeded, resident on cuda:0 before the first launch):

  linear_fwd / linear_bwd        minGRU linear scan, B=8 T=4096 D=1024, fp32
  linear_bf16_fwd / _bwd         minGRU linear scan, B=4 T=8192 D=4096, bf16 a, b
                                 (1/16 of the 2^31-element workload, same tiles)
  mingru_bf16_fwd / _bwd         fused minGRU gate + scan, B=4 T=8192 D=4096, bf16 x1, x2,
                                 forward without A, backward without gA, bf16 gradients
  varlen_fwd / varlen_bwd        packed ragged sequences (lengths 1..4096, seeded) of
                                 32768 rows x D=1024 in total, fp32, with start states
  log_fwd / log_bwd              minGRU log-space scan and its adjoint, B=8 T=2048 D=2048
  affine4_fwd / affine4_bwd      Haar affine scan, B=4 T=2048 n=64 k=v=4
  affine16_fwd / affine16_bwd    Haar affine scan, B=2 T=1024 n=32 k=v=16
  angle_fwd / angle_bwd          angle-fused scan, B=16 T=512 n=256 k=16 R=4 (a quarter of
                                 the bench's T; each input larger than L2)

Every case runs its op `repeats` times (default 3) after one set-up call of
the forward op where the backward needs the forward's outputs.  Each input is
larger than L2 except for the affine cases (134 MB and 268 MB in total).
"""
from __future__ import annotations

import sys

import torch

import linear_recurrence_scans_gb300 as mg
from linear_recurrence_scans_gb300 import workloads as wl

CASES = ("linear_fwd", "linear_bwd", "linear_bf16_fwd", "linear_bf16_bwd", "log_fwd", "log_bwd",
         "affine4_fwd", "affine4_bwd", "affine16_fwd", "affine16_bwd", "mingru_bf16_fwd",
         "mingru_bf16_bwd", "varlen_fwd", "varlen_bwd", "angle_fwd", "angle_bwd")


def main(argv):
    if not argv or argv[0] not in CASES:
        print(__doc__)
        return 2
    case = argv[0]
    reps = int(argv[1]) if len(argv) > 1 else 3
    dev = torch.device("cuda", 0)
    mg.load()
    if case.startswith("angle"):
        th, sc, ga, bv, h0, perm, sgn, p2p, go = wl.angle_inputs(16, 512, 256, 4, 16, seed=0,
                                                                 device=dev)
        h = mg.angle_scan_fwd(th, sc, ga, bv, h0, perm, sgn, p2p)
        outs = tuple(torch.empty_like(x) for x in (th, sc, ga, bv, h0))
        for _ in range(reps):
            if case.endswith("fwd"):
                mg.angle_scan_fwd(th, sc, ga, bv, h0, perm, sgn, p2p, out=h)
            else:
                mg.angle_scan_bwd(th, sc, ga, h0, h, go, perm, sgn, p2p, out=outs)
    elif case.startswith("mingru"):
        x1, x2, _, gBc = wl.mingru_x(4, 8192, 4096, seed=0, device=dev, in_dtype=torch.bfloat16)
        _, Bc = mg.mingru_scan_fwd(x1, x2, want_A=False)
        dx1, dx2 = torch.empty_like(x1), torch.empty_like(x1)
        for _ in range(reps):
            if case.endswith("fwd"):
                mg.mingru_scan_fwd(x1, x2, want_A=False, out=(None, Bc))
            else:
                mg.mingru_scan_bwd(x1, x2, None, Bc, None, gBc, grad_dtype=torch.bfloat16,
                                   out=(dx1, dx2))
    elif case.startswith("varlen"):
        import numpy as np
        rng = np.random.default_rng(7)
        lens = []
        while sum(lens) < 32768:
            lens.append(int(min(rng.integers(1, 4097), 32768 - sum(lens))))
        cu = torch.as_tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int64,
                             device=dev)
        a, b, gA, gH = (x[0] for x in wl.mingru_linear(1, 32768, 1024, seed=0, device=dev))
        h0 = torch.randn(len(lens), 1024, device=dev, generator=torch.Generator(dev).manual_seed(4))
        A, H = mg.linear_scan_varlen_fwd(a, b, cu, h0)
        da, db, dh0 = torch.empty_like(A), torch.empty_like(A), torch.empty_like(h0)
        for _ in range(reps):
            if case.endswith("fwd"):
                mg.linear_scan_varlen_fwd(a, b, cu, h0, out=(A, H))
            else:
                mg.linear_scan_varlen_bwd(a, cu, A, H, gA, gH, h0, out=(da, db, dh0))
    elif case.startswith("linear"):
        bf16 = "bf16" in case
        shape = (4, 8192, 4096) if bf16 else (8, 4096, 1024)
        a, b, gA, gBc = wl.mingru_linear(*shape, seed=0, device=dev,
                                         in_dtype=torch.bfloat16 if bf16 else torch.float32)
        A, Bc = mg.linear_scan_fwd(a, b)
        da, db = torch.empty_like(A), torch.empty_like(A)
        for _ in range(reps):
            if case.endswith("fwd"):
                mg.linear_scan_fwd(a, b, out=(A, Bc))
            else:
                mg.linear_scan_bwd(a, A, Bc, gA, gBc, out=(da, db))
    elif case.startswith("log"):
        lc, lv = wl.mingru_log(8, 2048, 2048, seed=0, device=dev)
        h = mg.parallel_scan_log_fwd(lc, lv)
        gh = torch.randn(lc.shape, device=dev, generator=torch.Generator(dev).manual_seed(1))
        dlc, dlv = torch.empty_like(lc), torch.empty_like(lv)
        for _ in range(reps):
            if case == "log_fwd":
                mg.parallel_scan_log_fwd(lc, lv, out=h)
            else:
                mg.parallel_scan_log_bwd(lc, lv, h, gh, out=(dlc, dlv))
    else:
        k = 4 if case.startswith("affine4") else 16
        shape = (4, 2048, 64) if k == 4 else (2, 1024, 32)
        A, Bm, gA, gB = wl.haar_affine(*shape, k, k, seed=0, device=dev)
        Abar, Bbar = mg.affine_scan_fwd(A, Bm)
        dA, dB = torch.empty_like(A), torch.empty_like(Bm)
        for _ in range(reps):
            if case.endswith("fwd"):
                mg.affine_scan_fwd(A, Bm, out=(Abar, Bbar))
            else:
                mg.affine_scan_bwd(A, Abar, Bbar, gA, gB, out=(dA, dB))
    torch.cuda.synchronize(dev)
    mg.workspace_status()
    print(f"ok {case} x{reps}")
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
