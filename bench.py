"""Benchmark of the minGRU scan library on one or more GB300s.

One step = one pass of the scan hot path over one synthetic minGRU batch
(B=8, T=4096, D=1024, float32): mg_linear_scan_fwd then mg_linear_scan_bwd
(the backward consumes the forward's outputs, as in training).  The metric is
scan elements per second (B*T*D per step), whole job.  The other workloads
(log-space scan, k x k affine scans, the large bf16 run) are measured once per
run and reported under "per_workload".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same step on its own GPU with its
own batch (weak scaling, no data-path collective); the timed region is
bracketed by a barrier and the max elapsed time over ranks is used.
``--impl reference`` times the float64 CPU oracle instead, on a bounded
sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "mingru_linear_8x4096x1024"
B, T, D = 8, 4096, 1024
METRIC = "scan elements/s (B*T*D per fwd+bwd step)"
UNIT = "elements/s"
FWD_BYTES_PER_ELT = 16   # read a, b; write A, Bc (fp32)
BWD_BYTES_PER_ELT = 28   # read a, A, Bc, gA, gBc; write da, db (fp32)


# ------------------------------------------------------------- helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(elapsed_s: float, units: float, world_size: int):
    """(max elapsed over ranks, total units over ranks).  Collective when the
    process group is initialised (any backend); identity otherwise."""
    if world_size == 1 or not torch.distributed.is_initialized():
        return elapsed_s, units
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world_size: int):
    if world_size > 1 and torch.distributed.is_initialized():
        torch.distributed.barrier()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def source_hash() -> str:
    """Hash of the CUDA sources and public header: the key under which ncu
    traffic figures in profiles/ stay valid."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_recurrence_scans_gb300", "csrc")
    files = sorted(os.path.join(csrc, f) for f in os.listdir(csrc))
    files.append(os.path.join(ROOT, "include", "mg_scan.h"))
    for fn in files:
        with open(fn, "rb") as f:
            h.update(os.path.basename(fn).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` on the bench workload from the
    committed ncu summary, or None when the kernels changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_hash") != source_hash():
        return None
    k = rec.get("kernels", {}).get(kernel)
    return None if k is None else k.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------- our arm

def run_ours(args, ws_size, rank, local):
    import linear_recurrence_scans_gb300 as mg
    from linear_recurrence_scans_gb300 import workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    mg.load()
    stream = torch.cuda.current_stream(dev)

    # Two resident input sets, used alternately, so no step reads what the
    # previous one left in L2 (each input tensor alone is larger than L2).
    sets = []
    for s in range(2):
        a, b, gA, gBc = wl.mingru_linear(B, T, D, seed=1000 * rank + 10 * s, device=dev)
        sets.append((a, b, gA, gBc))
    A = torch.empty_like(sets[0][0])
    Bc = torch.empty_like(A)
    da = torch.empty_like(A)
    db = torch.empty_like(A)
    ws = mg.new_workspace(mg.linear_workspace_size(B, T, D), dev)

    def step(i, evs=None):
        a, b, gA, gBc = sets[i & 1]
        if evs is not None:
            evs[0].record(stream)
        mg.mg_linear_scan_fwd(a, b, out=(A, Bc), ws=ws)
        if evs is not None:
            evs[1].record(stream)
        mg.mg_linear_scan_bwd(a, A, Bc, gA, gBc, out=(da, db), ws=ws)
        if evs is not None:
            evs[2].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    mg.workspace_status(ws)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(ws_size)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t0.record(stream)
        for i in range(args.steps):
            step(i, evs[i])
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(ws_size)
    elapsed = t0.elapsed_time(t1) * 1e-3
    mg.workspace_status(ws)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in evs]

    n = B * T * D
    max_elapsed, total_units = aggregate(elapsed, float(n * args.steps), ws_size)
    value = total_units / max_elapsed

    peak, peak_kind = measured_peaks()
    fwd_avg = statistics.mean(fwd_ms) * 1e-3
    bwd_avg = statistics.mean(bwd_ms) * 1e-3
    dom = "bwd" if bwd_avg >= fwd_avg else "fwd"
    kname = "linear_scan_bwd" if dom == "bwd" else "linear_scan_fwd"
    algo = (BWD_BYTES_PER_ELT if dom == "bwd" else FWD_BYTES_PER_ELT) * n
    dur = bwd_avg if dom == "bwd" else fwd_avg
    achieved = algo / dur / 1e9
    roofline = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1),
                "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
                "traffic": profiled_traffic(kname),
                "algorithmic_bytes_per_launch": algo,
                "fwd": {"avg_ms": round(fwd_avg * 1e3, 4),
                        "GB_s": round(FWD_BYTES_PER_ELT * n / fwd_avg / 1e9, 1),
                        "frac": round(FWD_BYTES_PER_ELT * n / fwd_avg / 1e9 / peak, 4)},
                "bwd": {"avg_ms": round(bwd_avg * 1e3, 4),
                        "GB_s": round(BWD_BYTES_PER_ELT * n / bwd_avg / 1e9, 1),
                        "frac": round(BWD_BYTES_PER_ELT * n / bwd_avg / 1e9 / peak, 4)}}

    e2e = run_e2e(mg, sets[0], dev, stream, args, ws, ws_size)
    extra = run_extra(mg, dev, peak) if (rank == 0 and not args.no_extra) else None
    cpu = cpu_baseline() if (rank == 0 and ws_size == 1 and not args.no_cpu) else None

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_size,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": max_elapsed / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "T": T, "D": D,
                   "ops": ["mg_linear_scan_fwd", "mg_linear_scan_bwd"],
                   "inputs": "minGRU gate: a = 1 - sigmoid(x1), b = sigmoid(x1) g(x2), "
                             "gA, gBc ~ N(0,1); seeded",
                   "l2": "inputs larger than L2 (each 134 MB tensor > 129 MB L2), two "
                         "resident input sets alternated between steps; no flush",
                   "parallelism": f"replicas x{ws_size} (channels/batches independent)"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": 2 * args.steps, "clocks": clk.summary(),
    }
    if extra is not None:
        line["per_workload"] = extra
    return line


def run_e2e(mg, inputs, dev, stream, args, ws, ws_size):
    """Same metric through the public API with host buffers: each step copies
    a, b, gA, gBc from pinned host memory, runs fwd + bwd and copies A, Bc,
    da, db back to pinned host memory.  Steps are pipelined the way a caller
    streaming batches would: copies in, compute and copies out run on three
    streams over two device buffer sets, ordered by events, so step i's
    copy-out overlaps step i+1's copy-in and compute.  The timed region spans
    every step's copies and kernels."""
    host_in = [x.cpu().pin_memory() for x in inputs]
    host_out = [[torch.empty(inputs[0].shape, dtype=torch.float32).pin_memory() for _ in range(4)]
                for _ in range(2)]
    bi = sum(x.numel() * x.element_size() for x in host_in)
    bo = sum(x.numel() * x.element_size() for x in host_out[0])
    dev_in = [[torch.empty_like(x, device=dev) for x in host_in] for _ in range(2)]
    dev_out = [[torch.empty(inputs[0].shape, dtype=torch.float32, device=dev) for _ in range(4)]
               for _ in range(2)]
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()  # noqa: E731
    k = max(3, min(args.steps, 20))

    def run(nsteps):
        done_cmp, done_out = [None, None], [None, None]
        for i in range(nsteps):
            j = i % 2
            with torch.cuda.stream(s_in):          # inputs of buffer j are free
                if done_cmp[j] is not None:
                    s_in.wait_event(done_cmp[j])
                for d, h in zip(dev_in[j], host_in):
                    d.copy_(h, non_blocking=True)
                e_in = ev()
                e_in.record(s_in)
            with torch.cuda.stream(s_cmp):         # outputs of buffer j are free
                s_cmp.wait_event(e_in)
                if done_out[j] is not None:
                    s_cmp.wait_event(done_out[j])
                a, b, gA, gBc = dev_in[j]
                A, Bc, da, db = dev_out[j]
                mg.mg_linear_scan_fwd(a, b, out=(A, Bc), ws=ws)
                mg.mg_linear_scan_bwd(a, A, Bc, gA, gBc, out=(da, db), ws=ws)
                done_cmp[j] = ev()
                done_cmp[j].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_cmp[j])
                for h, d in zip(host_out[j], dev_out[j]):
                    h.copy_(d, non_blocking=True)
                done_out[j] = ev()
                done_out[j].record(s_out)

    run(3)
    torch.cuda.synchronize(dev)
    barrier(ws_size)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    t0.record(s_in)
    run(k)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_cmp)
    t1.record(s_out)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - w0
    el, units = aggregate(max(t0.elapsed_time(t1) * 1e-3, wall), float(B * T * D * k), ws_size)
    return {"value": units / el, "unit": UNIT, "steps": k,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "ms_per_step": el / k * 1e3,
            "pipelining": "copy-in / compute / copy-out on three streams, two buffer sets"}


def _time_op(fn, iters, dev, flush):
    """Median CUDA-event time of fn() with an L2 flush before each repetition."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize(dev)
    ts = []
    for _ in range(iters):
        flush.zero_()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        e.synchronize()
        ts.append(s.elapsed_time(e) * 1e-3)
    return statistics.median(ts)


def run_extra(mg, dev, peak):
    """Each other workload once: median of a few repetitions, L2 flushed
    before each, CUDA events."""
    from linear_recurrence_scans_gb300 import workloads as wl
    out = {}
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    # log-space scan
    lc, lv = wl.mingru_log(16, 2048, 2048, seed=0, device=dev)
    h = torch.empty_like(lc)
    t = _time_op(lambda: mg.mg_log_scan_fwd(lc, lv, out=h), 10, dev, flush)
    n = lc.numel()
    byt = 12 * n + 4 * 16 * 2048
    out["mingru_log_16x2048x2048"] = {"op": "mg_log_scan_fwd", "ms": t * 1e3,
                                      "elements_per_s": n / t, "GB_s": byt / t / 1e9,
                                      "frac": byt / t / 1e9 / peak, "algorithmic_bytes": byt}
    # its adjoint: reads log_coeffs, log_values, h, gh; writes dlog_coeffs, dlog_values
    gh = torch.randn(lc.shape, device=dev, generator=torch.Generator(dev).manual_seed(1))
    dlc, dlv = torch.empty_like(lc), torch.empty_like(lv)
    t = _time_op(lambda: mg.mg_log_scan_bwd(lc, lv, h, gh, out=(dlc, dlv)), 10, dev, flush)
    byt = 24 * n + 8 * 16 * 2048
    out["mingru_log_bwd_16x2048x2048"] = {"op": "mg_log_scan_bwd", "ms": t * 1e3,
                                          "elements_per_s": n / t, "GB_s": byt / t / 1e9,
                                          "frac": byt / t / 1e9 / peak, "algorithmic_bytes": byt}
    del lc, lv, h, gh, dlc, dlv
    # affine scans
    fp32_peak_tflops = 152 * 128 * 2 * 2.07e9 / 1e12  # FFMA lanes x 2 flop x max SM clock
    for name, (Bq, Tq, nq, k, v) in (("haar_affine_4x2048x64_k4v4", (4, 2048, 64, 4, 4)),
                                     ("haar_affine_2x1024x32_k16v16", (2, 1024, 32, 16, 16))):
        A, Bm, gA, gB = wl.haar_affine(Bq, Tq, nq, k, v, seed=0, device=dev)
        Abar, Bbar = torch.empty_like(A), torch.empty_like(Bm)
        dA, dB = torch.empty_like(A), torch.empty_like(Bm)
        S = Bq * Tq * nq
        tf = _time_op(lambda: mg.mg_affine_scan_fwd(A, Bm, out=(Abar, Bbar)), 10, dev, flush)
        tb = _time_op(lambda: mg.mg_affine_scan_bwd(A, Abar, Bbar, gA, gB, out=(dA, dB)), 10,
                      dev, flush)
        fb, bb = S * 4 * 2 * (k * k + k * v), S * 4 * (4 * k * k + 3 * k * v)
        ff, bf = S * 2 * (k ** 3 + k * k * v), S * 4 * (k ** 3 + k * k * v)
        rf = max(fb / (peak * 1e9), ff / (fp32_peak_tflops * 1e12))
        rb = max(bb / (peak * 1e9), bf / (fp32_peak_tflops * 1e12))
        out[name] = {"op": "mg_affine_scan_fwd + mg_affine_scan_bwd",
                     "elements": S * k * v,
                     "fwd": {"ms": tf * 1e3, "elements_per_s": S * k * v / tf,
                             "GB_s": fb / tf / 1e9, "TFLOP_s": ff / tf / 1e12,
                             "roofline_frac": rf / tf},
                     "bwd": {"ms": tb * 1e3, "elements_per_s": S * k * v / tb,
                             "GB_s": bb / tb / 1e9, "TFLOP_s": bf / tb / 1e12,
                             "roofline_frac": rb / tb},
                     "roofline": "max(bytes / HBM peak, flops / FP32 FFMA peak "
                                 f"{fp32_peak_tflops:.1f} TFLOP/s at 2070 MHz)"}
        del A, Bm, gA, gB, Abar, Bbar, dA, dB
    # large bf16 linear scan (2^31 elements)
    Bq, Tq, Dq = 16, 32768, 4096
    a, b, gA, gBc = wl.mingru_linear(Bq, Tq, Dq, seed=0, device=dev, in_dtype=torch.bfloat16)
    A, Bc = mg.mg_linear_scan_fwd(a, b)
    da, db = torch.empty_like(A), torch.empty_like(A)
    n = a.numel()
    tf = _time_op(lambda: mg.mg_linear_scan_fwd(a, b, out=(A, Bc)), 5, dev, flush)
    tb = _time_op(lambda: mg.mg_linear_scan_bwd(a, A, Bc, gA, gBc, out=(da, db)), 5, dev, flush)
    out["mingru_linear_bf16_16x32768x4096"] = {
        "op": "mg_linear_scan_fwd + mg_linear_scan_bwd (bf16 a, b)", "elements": n,
        "fwd": {"ms": tf * 1e3, "elements_per_s": n / tf, "GB_s": 12 * n / tf / 1e9,
                "frac": 12 * n / tf / 1e9 / peak},
        "bwd": {"ms": tb * 1e3, "elements_per_s": n / tb, "GB_s": 26 * n / tb / 1e9,
                "frac": 26 * n / tb / 1e9 / peak},
        "step_elements_per_s": n / (tf + tb)}
    del a, b, gA, gBc, A, Bc, da, db, flush
    mg.workspace_status()
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------- CPU legs

def _oracle_step_on_sample(ncols: int, seed: int = 0):
    """Oracle fwd + bwd on `ncols` independent channels (all of T) of the
    workload: exact for those channels.  Returns (elements, seconds)."""
    import oracle
    from linear_recurrence_scans_gb300 import workloads as wl
    a, b, gA, gBc = wl.mingru_linear(1, T, ncols, seed=seed)
    a, b, gA, gBc = (x.double().numpy() for x in (a, b, gA, gBc))
    t0 = time.perf_counter()
    A, Bc = oracle.linear_scan_fwd(a, b)
    oracle.linear_scan_bwd(a, A, Bc, gA, gBc)
    return a.size, time.perf_counter() - t0


def cpu_baseline(target_s: float = 10.0):
    """The oracle as it stands (single-threaded C, float64) on a bounded
    sample: whole batch rows of the workload (all T, all D of one b), one
    after another (different seeds), until about `target_s` seconds of CPU
    work."""
    import oracle
    oracle.build()
    els, secs, reps = 0, 0.0, 0
    while secs < target_s and reps < 400:
        e, s = _oracle_step_on_sample(D, seed=reps)
        els += e
        secs += s
        reps += 1
    return {"value": els / secs, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{reps} x one batch row (T={T}, D={D}) of {WORKLOAD}, fwd+bwd, "
                      f"float64 C oracle, {secs:.1f} s"}


def run_reference(args, ws_size, rank):
    """--impl reference: the oracle on the host cores, each step a bounded
    sample of the workload (whole-T channel columns)."""
    import oracle
    oracle.build()
    # calibrate: size the per-step sample so the whole run stays within ~90 s
    e, s = _oracle_step_on_sample(64)
    per_col = s / 64
    budget = 90.0 / max(1, args.steps + args.warmup)
    ncols = int(max(8, min(D, budget / per_col)))
    for i in range(args.warmup):
        _oracle_step_on_sample(ncols, seed=i)
    els, secs = 0, 0.0
    for i in range(args.steps):
        e, s = _oracle_step_on_sample(ncols, seed=100 + i)
        els += e
        secs += s
    value = els / secs
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_size,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "T": T, "D": D,
                   "ops": ["oracle.linear_scan_fwd", "oracle.linear_scan_bwd"]},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{ncols} whole-T channels of {WORKLOAD} per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    ws_size, rank, local = dist_env()
    if ws_size > 1:
        torch.distributed.init_process_group(
            backend="nccl" if torch.cuda.is_available() else "gloo")
    try:
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps(run_reference(args, ws_size, rank)), flush=True)
            return
        line = run_ours(args, ws_size, rank, local)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        if ws_size > 1 and torch.distributed.is_initialized():
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
