"""Parity of every op against the float64 oracle in one process, run by
test_engines_gpu.py as a child process with MGSCAN_ENGINE set.

The library reads MGSCAN_ENGINE once per process, so each engine choice
("chunked": every op on the chunk engine; "stream": every op that has a
persistent streaming variant on it) needs a process of its own.  Shapes are
ragged in time and channels and span several tiles and chunks.

    python tests/engine_check.py        # prints one line per case, exit 1 on a failure
"""
from __future__ import annotations

import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import torch  # noqa: E402

import linear_recurrence_scans_gb300 as mg  # noqa: E402
import oracle  # noqa: E402
from linear_recurrence_scans_gb300 import workloads as wl  # noqa: E402
from parity import (TOL_BF16, TOL_F32, affine_bwd_errors, affine_fwd_errors,  # noqa: E402
                    linear_bwd_errors, linear_fwd_errors, log_bwd_errors, log_fwd_errors)

DEV = "cuda"


def main() -> int:
    mg.load()
    failed = []

    def report(name, errs, tol):
        worst = max(errs.values())
        ok = worst <= tol
        print(f"{name:40s} worst {worst:.3g} {'ok' if ok else 'FAIL'}", flush=True)
        if not ok:
            failed.append(name)

    for shape in ((3, 517, 300), (1, 4099, 8), (2, 1500, 512)):
        for dt, tol in ((torch.float32, TOL_F32), (torch.bfloat16, TOL_BF16)):
            a, b, gA, gBc = wl.mingru_linear(*shape, seed=21, in_dtype=dt)
            A, Bc = mg.linear_scan_fwd(a.to(DEV), b.to(DEV))
            report(f"linear_fwd {shape} {dt}", linear_fwd_errors(a, b, A, Bc), tol)
            rA, rBc = oracle.linear_scan_fwd(a, b)
            A32, Bc32 = torch.from_numpy(rA).float(), torch.from_numpy(rBc).float()
            da, db = mg.linear_scan_bwd(a.to(DEV), A32.to(DEV), Bc32.to(DEV), gA.to(DEV), gBc.to(DEV))
            report(f"linear_bwd {shape} {dt}", linear_bwd_errors(a, A32, Bc32, gA, gBc, da, db), tol)
        lc, lv = wl.mingru_log(*shape, seed=22)
        h = mg.parallel_scan_log_fwd(lc.to(DEV), lv.to(DEV))
        report(f"log_fwd {shape}", log_fwd_errors(lc, lv, h), TOL_F32)
        gh = torch.randn(lc.shape, generator=torch.Generator().manual_seed(26))
        h32 = torch.from_numpy(oracle.log_scan_fwd(lc, lv)).float()
        dlc, dlv = mg.parallel_scan_log_bwd(lc.to(DEV), lv.to(DEV), h32.to(DEV), gh.to(DEV))
        report(f"log_bwd {shape}", log_bwd_errors(lc, lv, gh, dlc, dlv), TOL_F32)

    for (B, T, n), k, v in (((2, 333, 5), 2, 2), ((2, 333, 5), 4, 4), ((1, 700, 3), 4, 16),
                            ((2, 200, 3), 8, 8), ((2, 150, 3), 16, 16)):
        A, Bm, gA, gB = wl.haar_affine(B, T, n, k, v, seed=23)
        Abar, Bbar = mg.affine_scan_fwd(A.to(DEV), Bm.to(DEV))
        report(f"affine_fwd {(B, T, n)} k{k} v{v}", affine_fwd_errors(A, Bm, Abar, Bbar), TOL_F32)
        rAbar, rBbar = oracle.affine_scan_fwd(A, Bm)
        Ab32, Bb32 = torch.from_numpy(rAbar).float(), torch.from_numpy(rBbar).float()
        dA, dB = mg.affine_scan_bwd(A.to(DEV), Ab32.to(DEV), Bb32.to(DEV), gA.to(DEV), gB.to(DEV))
        report(f"affine_bwd {(B, T, n)} k{k} v{v}",
               affine_bwd_errors(A, Ab32, Bb32, gA, gB, dA, dB), TOL_F32)

    mg.workspace_status()
    print("engine", os.environ.get("MGSCAN_ENGINE", "auto"), "failed:", failed, flush=True)
    return 1 if failed else 0


if __name__ == "__main__":
    sys.exit(main())
