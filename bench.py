"""Benchmark of the minGRU scan library on one or more GB300s.

One step = one pass of the scan hot path over one synthetic minGRU batch,
the largest workload: B=16, T=32768, D=4096 (2^31 elements), a and b in
bf16, float32 accumulation and float32 outputs: mg_linear_scan_fwd then
mg_linear_scan_bwd (the backward consumes the forward's outputs, as in
training).  The metric is scan elements per second (B*T*D per step), whole
job.  The other workloads (the float32 minGRU batch 8x4096x1024, the
log-space scan and its adjoint, the k x k affine scans) are measured once per
run and reported under "per_workload".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same step on its own GPU with its
own batch (weak scaling, no data-path collective); the timed region is
bracketed by a barrier and the max elapsed time over ranks is used.
``--impl reference`` times the float64 CPU oracle instead, on a bounded
sample of the same workload (whole-T channel columns), on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "mingru_linear_bf16_16x32768x4096"
B, T, D = 16, 32768, 4096
METRIC = "scan elements/s (B*T*D per fwd+bwd step)"
UNIT = "elements/s"
FWD_BYTES_PER_ELT = 12   # read a, b (bf16); write A, Bc (fp32)
BWD_BYTES_PER_ELT = 26   # read a (bf16), A, Bc, gA, gBc; write da, db (fp32)


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
    committed ncu summary (scaled from the captured case to a full launch by
    the elements processed, as the record states), or None when the kernels
    changed since the capture."""
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
    """nvidia-smi clock/throttle samples every `period_ms` while active."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)   # let the first samples arrive before the timed work
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

    def summary(self, window: str):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for *_, r in rows for i, v in enumerate(r) if v == "Active"})
        # samples under load: the power draw separates them from the idle edges
        pmax = max(r[2] for r in rows)
        load = [r for r in rows if r[2] >= 0.5 * pmax] or rows
        return {"sm_mhz": statistics.median(r[0] for r in load),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(load),
                "power_w_max": pmax, "period_ms": self.period, "window": window}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def events_ms(pairs):
    return [s.elapsed_time(e) for s, e in pairs]


# ------------------------------------------------------------- our arm

def run_ours(args, ws_size, rank, local):
    import linear_recurrence_scans_gb300 as mg
    from linear_recurrence_scans_gb300 import workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    mg.load()
    stream = torch.cuda.current_stream(dev)

    # One resident batch: every input tensor (4.3 GB bf16, 8.6 GB fp32) is
    # far larger than L2, so no step finds the previous one's data there.
    a, b, gA, gBc = wl.mingru_linear(B, T, D, seed=1000 * rank, device=dev,
                                     in_dtype=torch.bfloat16)
    A = torch.empty(a.shape, dtype=torch.float32, device=dev)
    Bc, da, db = torch.empty_like(A), torch.empty_like(A), torch.empty_like(A)
    ws = mg.new_workspace(mg.linear_workspace_size(B, T, D), dev)

    def step(evs=None):
        if evs is not None:
            evs[0].record(stream)
        mg.mg_linear_scan_fwd(a, b, out=(A, Bc), ws=ws)
        if evs is not None:
            evs[1].record(stream)
        mg.mg_linear_scan_bwd(a, A, Bc, gA, gBc, out=(da, db), ws=ws)
        if evs is not None:
            evs[2].record(stream)

    for _ in range(args.warmup):
        step()
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
            step(evs[i])
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(ws_size)
    elapsed = t0.elapsed_time(t1) * 1e-3
    mg.workspace_status(ws)
    fwd_ms = events_ms((e[0], e[1]) for e in evs)
    bwd_ms = events_ms((e[1], e[2]) for e in evs)

    n = B * T * D
    max_elapsed, total_units = aggregate(elapsed, float(n * args.steps), ws_size)
    value = total_units / max_elapsed

    peak, peak_kind = measured_peaks()
    fwd_avg = statistics.mean(fwd_ms) * 1e-3
    bwd_avg = statistics.mean(bwd_ms) * 1e-3
    dom = "bwd" if bwd_avg >= fwd_avg else "fwd"
    kname = "linear_scan_bwd_bf16" if dom == "bwd" else "linear_scan_fwd_bf16"
    algo = (BWD_BYTES_PER_ELT if dom == "bwd" else FWD_BYTES_PER_ELT) * n
    dur = bwd_avg if dom == "bwd" else fwd_avg
    achieved = algo / dur / 1e9

    def leg(bpe, avg, ms):
        return {"avg_ms": round(avg * 1e3, 4), "median_ms": round(statistics.median(ms), 4),
                "GB_s": round(bpe * n / avg / 1e9, 1),
                "frac": round(bpe * n / avg / 1e9 / peak, 4),
                "algorithmic_bytes_per_launch": bpe * n,
                "traffic": profiled_traffic("linear_scan_fwd_bf16" if bpe == FWD_BYTES_PER_ELT
                                            else "linear_scan_bwd_bf16")}

    roofline = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1),
                "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json), burst copy",
                "traffic": profiled_traffic(kname),
                "algorithmic_bytes_per_launch": algo,
                "fwd": leg(FWD_BYTES_PER_ELT, fwd_avg, fwd_ms),
                "bwd": leg(BWD_BYTES_PER_ELT, bwd_avg, bwd_ms)}
    clocks = clk.summary(f"timed region: {args.steps} steps, {max_elapsed * 1e3:.1f} ms")
    del A, Bc, da, db, ws
    inputs = (a, b, gA, gBc)
    del a, b, gA, gBc

    e2e = run_e2e(mg, inputs, dev, args, ws_size)
    del inputs
    torch.cuda.empty_cache()
    extra = run_extra(mg, dev, peak) if (rank == 0 and not args.no_extra) else None
    cpu = cpu_baseline() if (rank == 0 and ws_size == 1 and not args.no_cpu) else None

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_size,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": max_elapsed / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, f32 accumulation and out",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "T": T, "D": D,
                   "ops": ["mg_linear_scan_fwd", "mg_linear_scan_bwd"],
                   "inputs": "minGRU gate: a = 1 - sigmoid(x1), b = sigmoid(x1) g(x2) rounded "
                             "to bf16; gA, gBc ~ N(0,1) float32; seeded, generated on the GPU",
                   "l2": "inputs larger than L2 (4.3 GB bf16 and 8.6 GB fp32 tensors against "
                         "a 129 MB L2); no flush",
                   "parallelism": f"replicas x{ws_size} (channels/batches independent)"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": 2 * args.steps, "clocks": clocks,
    }
    if extra is not None:
        line["per_workload"] = extra
    return line


def link_rates(dev, nbytes=1 << 30):
    """Raw pinned host <-> device copy rates (GB/s): each direction alone and
    both at once on two streams; median of 5."""
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn):
        ts = []
        for _ in range(6):
            torch.cuda.synchronize(dev)
            w = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            ts.append(time.perf_counter() - w)
        return statistics.median(ts[1:])

    def h2d():
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            h_out.copy_(d_out, non_blocking=True)

    def both():
        h2d()
        d2h()

    th, td, tb = timed(h2d), timed(d2h), timed(both)
    return {"h2d_GB_s": round(nbytes / th / 1e9, 1), "d2h_GB_s": round(nbytes / td / 1e9, 1),
            "bidirectional_GB_s_each": round(nbytes / tb / 1e9, 1),
            "how": "1 GiB pinned copies, median of 5, wall clock around synchronize"}


NBUF = 3   # row buffers in the end-to-end pipeline (device and pinned host each)


def run_e2e(mg, inputs, dev, args, ws_size):
    """Same metric through the public API with host buffers.  A caller streams
    the batch through the GPU one batch row (T x D = 2^27 elements) at a time:
    per row, a and b (bf16) and gA, gBc (fp32) are copied from pinned host
    memory, fwd + bwd run on the row, and A, Bc, da, db are copied back to
    pinned host memory.  Rows are pipelined on three streams (copy in,
    compute, copy out) over NBUF device buffer sets and NBUF pinned host
    buffer sets (the host ring a data loader would use), so host memory
    stays at NBUF rows.  A step is all B rows; the timed region spans every
    row's copies and kernels."""
    a, b, gA, gBc = inputs
    host_in = [[x[r].cpu().pin_memory() for x in (a, b, gA, gBc)] for r in range(NBUF)]
    row_shape = (1, T, D)
    host_out = [[torch.empty(row_shape, dtype=torch.float32).pin_memory() for _ in range(4)]
                for _ in range(NBUF)]
    bi_row = sum(x.numel() * x.element_size() for x in host_in[0])
    bo_row = sum(x.numel() * x.element_size() for x in host_out[0])
    dev_in = [[torch.empty(row_shape, dtype=x.dtype, device=dev) for x in host_in[0]]
              for _ in range(NBUF)]
    dev_out = [[torch.empty(row_shape, dtype=torch.float32, device=dev) for _ in range(4)]
               for _ in range(NBUF)]
    ws = mg.new_workspace(mg.linear_workspace_size(1, T, D), dev)
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()  # noqa: E731
    k = 3
    rate = link_rates(dev)

    def run(nsteps):
        done_cmp, done_out = [None] * NBUF, [None] * NBUF
        for i in range(nsteps * B):
            j = i % NBUF
            with torch.cuda.stream(s_in):          # inputs of buffer j are free
                if done_cmp[j] is not None:
                    s_in.wait_event(done_cmp[j])
                for d_, h in zip(dev_in[j], host_in[j]):
                    d_.copy_(h.view(row_shape), non_blocking=True)
                e_in = ev()
                e_in.record(s_in)
            with torch.cuda.stream(s_cmp):         # outputs of buffer j are free
                s_cmp.wait_event(e_in)
                if done_out[j] is not None:
                    s_cmp.wait_event(done_out[j])
                ra, rb, rgA, rgB = dev_in[j]
                rA, rBc, rda, rdb = dev_out[j]
                mg.mg_linear_scan_fwd(ra, rb, out=(rA, rBc), ws=ws)
                mg.mg_linear_scan_bwd(ra, rA, rBc, rgA, rgB, out=(rda, rdb), ws=ws)
                done_cmp[j] = ev()
                done_cmp[j].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_cmp[j])
                for h, d_ in zip(host_out[j], dev_out[j]):
                    h.copy_(d_, non_blocking=True)
                done_out[j] = ev()
                done_out[j].record(s_out)

    run(1)
    torch.cuda.synchronize(dev)
    mg.workspace_status(ws)
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
    mg.workspace_status(ws)
    el, units = aggregate(max(t0.elapsed_time(t1) * 1e-3, wall), float(B * T * D * k), ws_size)
    bi, bo = bi_row * B, bo_row * B
    ms = el / k * 1e3
    return {"value": units / el, "unit": UNIT, "steps": k,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "ms_per_step": ms,
            "copy_GB_s_each_way": {"h2d": round(bi / (ms * 1e-3) / 1e9, 1),
                                   "d2h": round(bo / (ms * 1e-3) / 1e9, 1)},
            "link": rate,
            "link_bound_ms_per_step": round(max(bi, bo) / (rate["bidirectional_GB_s_each"] * 1e9)
                                            * 1e3, 1),
            "pipelining": f"{B} batch rows per step; copy-in / compute / copy-out on three "
                          f"streams, {NBUF} device and {NBUF} pinned host row buffers"}


def _time_op(fn, iters, dev, flush):
    """Median CUDA-event time of fn() with an L2 flush before each repetition:
    the flush buffer (larger than L2) is written, then read back, so that L2
    holds neither the op's inputs nor dirty lines whose write-back would be
    charged to the op."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize(dev)
    ts = []
    for _ in range(iters):
        flush.zero_()
        flush.sum(dtype=torch.int64)
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        e.synchronize()
        ts.append(s.elapsed_time(e) * 1e-3)
    return statistics.median(ts)


def run_extra(mg, dev, peak):
    """Each other workload once: median of several repetitions, L2 flushed
    before each, CUDA events."""
    from linear_recurrence_scans_gb300 import workloads as wl
    out = {}
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    # the float32 minGRU batch
    Bq, Tq, Dq = 8, 4096, 1024
    a, b, gA, gBc = wl.mingru_linear(Bq, Tq, Dq, seed=0, device=dev)
    A, Bc = mg.mg_linear_scan_fwd(a, b)
    da, db = torch.empty_like(A), torch.empty_like(A)
    n = a.numel()
    tf = _time_op(lambda: mg.mg_linear_scan_fwd(a, b, out=(A, Bc)), 20, dev, flush)
    tb = _time_op(lambda: mg.mg_linear_scan_bwd(a, A, Bc, gA, gBc, out=(da, db)), 20, dev, flush)
    out["mingru_linear_8x4096x1024"] = {
        "op": "mg_linear_scan_fwd + mg_linear_scan_bwd (fp32)", "elements": n,
        "fwd": {"ms": tf * 1e3, "elements_per_s": n / tf, "GB_s": 16 * n / tf / 1e9,
                "frac": 16 * n / tf / 1e9 / peak},
        "bwd": {"ms": tb * 1e3, "elements_per_s": n / tb, "GB_s": 28 * n / tb / 1e9,
                "frac": 28 * n / tb / 1e9 / peak},
        "step_elements_per_s": n / (tf + tb)}
    # the same batch from start states h0 (B, D)
    h0 = torch.randn(Bq, Dq, device=dev, generator=torch.Generator(dev).manual_seed(3))
    dh0 = torch.empty_like(h0)
    tf = _time_op(lambda: mg.mg_linear_scan_h0_fwd(a, b, h0, out=(A, Bc)), 20, dev, flush)
    tb = _time_op(lambda: mg.mg_linear_scan_h0_bwd(a, h0, A, Bc, gA, gBc, out=(da, db, dh0)), 20,
                  dev, flush)
    fb, bb = 16 * n + 4 * h0.numel(), 28 * n + 8 * h0.numel()
    out["mingru_linear_h0_8x4096x1024"] = {
        "op": "mg_linear_scan_h0_fwd + mg_linear_scan_h0_bwd (fp32, start states h0)",
        "elements": n,
        "fwd": {"ms": tf * 1e3, "GB_s": fb / tf / 1e9, "frac": fb / tf / 1e9 / peak},
        "bwd": {"ms": tb * 1e3, "GB_s": bb / tb / 1e9, "frac": bb / tb / 1e9 / peak}}
    # the same elements as one packed batch of ragged sequences (lengths
    # 1..4096, seeded), each from its own start state
    rng = np.random.default_rng(7)
    lens = []
    while sum(lens) < Bq * Tq:
        lens.append(int(min(rng.integers(1, 4097), Bq * Tq - sum(lens))))
    cu = torch.as_tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int64, device=dev)
    nseq = len(lens)
    hs = torch.randn(nseq, Dq, device=dev, generator=torch.Generator(dev).manual_seed(4))
    dhs = torch.empty_like(hs)
    pa, pb = a.reshape(Bq * Tq, Dq), b.reshape(Bq * Tq, Dq)
    pA, pH = A.reshape(Bq * Tq, Dq), Bc.reshape(Bq * Tq, Dq)
    pgA, pgH = gA.reshape(Bq * Tq, Dq), gBc.reshape(Bq * Tq, Dq)
    pda, pdb = da.reshape(Bq * Tq, Dq), db.reshape(Bq * Tq, Dq)
    tf = _time_op(lambda: mg.mg_linear_scan_varlen_fwd(pa, pb, cu, hs, out=(pA, pH)), 20, dev,
                  flush)
    tb = _time_op(lambda: mg.mg_linear_scan_varlen_bwd(pa, cu, pA, pH, pgA, pgH, hs,
                                                       out=(pda, pdb, dhs)), 20, dev, flush)
    fb = 16 * n + 4 * hs.numel() + 8 * (nseq + 1)
    bb = 28 * n + 8 * hs.numel() + 8 * (nseq + 1)
    out["mingru_varlen_packed_32768x1024"] = {
        "op": "mg_linear_scan_varlen_fwd + _bwd (fp32, packed ragged sequences with start states)",
        "elements": n, "sequences": nseq,
        "fwd": {"ms": tf * 1e3, "GB_s": fb / tf / 1e9, "frac": fb / tf / 1e9 / peak},
        "bwd": {"ms": tb * 1e3, "GB_s": bb / tb / 1e9, "frac": bb / tb / 1e9 / peak}}
    del a, b, gA, gBc, A, Bc, da, db, h0, dh0, hs, dhs
    # the fused minGRU gate + scan, as a minGRU layer trains: forward without
    # A, backward without gA (the loss depends on h = Bc only)
    for name, (Bq, Tq, Dq, xdt) in (("mingru_fused_8x4096x1024", (8, 4096, 1024, torch.float32)),
                                    ("mingru_fused_bf16_16x32768x4096",
                                     (16, 32768, 4096, torch.bfloat16))):
        x1, x2, _, gBc = wl.mingru_x(Bq, Tq, Dq, seed=0, device=dev, in_dtype=xdt)
        _, Bc = mg.mingru_scan_fwd(x1, x2, want_A=False)
        dx1, dx2 = torch.empty_like(x1), torch.empty_like(x1)
        n = x1.numel()
        xs = x1.element_size()
        reps = 20 if n < (1 << 28) else 5
        tf = _time_op(lambda: mg.mingru_scan_fwd(x1, x2, want_A=False, out=(None, Bc)), reps,
                      dev, flush)
        tb = _time_op(lambda: mg.mingru_scan_bwd(x1, x2, None, Bc, None, gBc, grad_dtype=xdt,
                                                 out=(dx1, dx2)), reps, dev, flush)
        fb = (2 * xs + 4) * n          # read x1, x2; write Bc
        bb = (2 * xs + 8 + 2 * xs) * n  # read x1, x2, Bc, gBc; write dx1, dx2
        out[name] = {
            "op": "mg_mingru_scan_fwd (no A) + mg_mingru_scan_bwd (no gA), gradients in the "
                  "input dtype", "elements": n,
            "fwd": {"ms": tf * 1e3, "elements_per_s": n / tf, "GB_s": fb / tf / 1e9,
                    "frac": fb / tf / 1e9 / peak, "algorithmic_bytes": fb},
            "bwd": {"ms": tb * 1e3, "elements_per_s": n / tb, "GB_s": bb / tb / 1e9,
                    "frac": bb / tb / 1e9 / peak, "algorithmic_bytes": bb},
            "step_elements_per_s": n / (tf + tb)}
        del x1, x2, gBc, Bc, dx1, dx2
        torch.cuda.empty_cache()
    # the angle-fused scan (Kernel 4): 4096 sequences of k = 16, R = 4 layers
    Bq, Tq, nq, R, k = 16, 2048, 256, 4, 16
    th, sc, ga, bv, h0, perm, sgn, p2p, go = wl.angle_inputs(Bq, Tq, nq, R, k, seed=0, device=dev)
    h = mg.angle_scan_fwd(th, sc, ga, bv, h0, perm, sgn, p2p)
    outs = tuple(torch.empty_like(x) for x in (th, sc, ga, bv, h0))
    tf = _time_op(lambda: mg.angle_scan_fwd(th, sc, ga, bv, h0, perm, sgn, p2p, out=h), 10, dev,
                  flush)
    tb = _time_op(lambda: mg.angle_scan_bwd(th, sc, ga, h0, h, go, perm, sgn, p2p, out=outs), 10,
                  dev, flush)
    S = Bq * Tq * nq
    fb = S * 4 * (R * k // 2 + 2 + 2 * k) + h0.numel() * 4          # theta, scale, gamma, b, h
    bb = S * 4 * (2 * (R * k // 2) + 4 + 3 * k) + 2 * h0.numel() * 4  # + out, grad_out; d*
    out["angle_16x2048x256_k16_R4"] = {
        "op": "mg_angle_scan_fwd + mg_angle_scan_bwd (has_scale, has_decay)",
        "elements": S * k,
        "fwd": {"ms": tf * 1e3, "elements_per_s": S * k / tf, "GB_s": fb / tf / 1e9,
                "frac": fb / tf / 1e9 / peak, "algorithmic_bytes": fb},
        "bwd": {"ms": tb * 1e3, "elements_per_s": S * k / tb, "GB_s": bb / tb / 1e9,
                "frac": bb / tb / 1e9 / peak, "algorithmic_bytes": bb}}
    del th, sc, ga, bv, h0, go, h, outs
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
        Am, Bm, gAm, gBm = wl.haar_affine(Bq, Tq, nq, k, v, seed=0, device=dev)
        Abar, Bbar = torch.empty_like(Am), torch.empty_like(Bm)
        dA, dB = torch.empty_like(Am), torch.empty_like(Bm)
        S = Bq * Tq * nq
        tf = _time_op(lambda: mg.mg_affine_scan_fwd(Am, Bm, out=(Abar, Bbar)), 10, dev, flush)
        tb = _time_op(lambda: mg.mg_affine_scan_bwd(Am, Abar, Bbar, gAm, gBm, out=(dA, dB)), 10,
                      dev, flush)
        fb, bb = S * 4 * 2 * (k * k + k * v), S * 4 * (4 * k * k + 3 * k * v)
        ff, bf = S * 2 * (k ** 3 + k * k * v), S * 4 * (k ** 3 + k * k * v)
        rf = max(fb / (peak * 1e9), ff / (fp32_peak_tflops * 1e12))
        rb = max(bb / (peak * 1e9), bf / (fp32_peak_tflops * 1e12))
        H0 = torch.randn(Bq, nq, k, v, device=dev, generator=torch.Generator(dev).manual_seed(5))
        dH0 = torch.empty_like(H0)
        tfh = _time_op(lambda: mg.mg_affine_scan_h0_fwd(Am, Bm, H0, out=(Abar, Bbar)), 10, dev,
                       flush)
        tbh = _time_op(lambda: mg.mg_affine_scan_h0_bwd(Am, H0, Abar, Bbar, gAm, gBm,
                                                        out=(dA, dB, dH0)), 10, dev, flush)
        out[name + "_h0"] = {"op": "mg_affine_scan_h0_fwd + mg_affine_scan_h0_bwd",
                             "fwd": {"ms": tfh * 1e3,
                                     "roofline_frac": (rf + H0.numel() * 4 / (peak * 1e9)) / tfh},
                             "bwd": {"ms": tbh * 1e3,
                                     "roofline_frac": (rb + H0.numel() * 8 / (peak * 1e9)) / tbh}}
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
        del Am, Bm, gAm, gBm, Abar, Bbar, dA, dB, H0, dH0
    del flush
    mg.workspace_status()
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------- CPU legs

SAMPLE_COLS = 128   # whole-T channel columns per oracle call


def _sample(seed: int, ncols: int = SAMPLE_COLS):
    """`ncols` independent whole-T channels of the workload (a, b rounded to
    bf16 as on the GPU, widened exactly to float64)."""
    from linear_recurrence_scans_gb300 import workloads as wl
    a, b, gA, gBc = wl.mingru_linear(1, T, ncols, seed=seed, in_dtype=torch.bfloat16)
    return tuple(np.ascontiguousarray(x.double().numpy()) for x in (a, b, gA, gBc))


def _oracle_fwd_bwd(sample):
    """The oracle's fwd + bwd on one sample; returns its elements."""
    import oracle
    a, b, gA, gBc = sample
    A, Bc = oracle.linear_scan_fwd(a, b)
    oracle.linear_scan_bwd(a, A, Bc, gA, gBc)
    return a.size


def _oracle_run(samples, threads: int, target_s: float):
    """Run the oracle over `samples` (cycled) on `threads` host threads until
    about `target_s` seconds have passed.  ctypes releases the GIL for the
    duration of each C call, so the threads run on separate cores.  Returns
    (elements, seconds, calls)."""
    stop = time.perf_counter() + target_s
    counts = [0] * threads
    calls = [0] * threads

    def worker(w):
        i = w
        while time.perf_counter() < stop:
            counts[w] += _oracle_fwd_bwd(samples[i % len(samples)])
            calls[w] += 1
            i += threads

    t0 = time.perf_counter()
    ths = [threading.Thread(target=worker, args=(w,)) for w in range(threads)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    return sum(counts), time.perf_counter() - t0, sum(calls)


def cpu_baseline(target_s: float = 10.0):
    """The oracle as it stands (sequential float64 C) on bounded samples of
    the workload: seeded whole-T channel columns (exact for those channels,
    which are independent).  One leg on one core, one leg on every host core
    (one oracle call per thread, each on its own sample)."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    samples = [_sample(seed) for seed in range(4)]
    e1, s1, c1 = _oracle_run(samples, 1, target_s)
    eN, sN, cN = _oracle_run(samples, cores, target_s)
    return {"value": e1 / s1, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{c1} oracle fwd+bwd calls on {SAMPLE_COLS} whole-T (T={T}) channel "
                      f"columns of {WORKLOAD} (4 seeded samples cycled), {s1:.1f} s on one core",
            "cpu_model": cpu_model(),
            "all_cores": {"value": eN / sN, "unit": UNIT, "cores": cores,
                          "sample": f"{cN} calls on {cores} threads, {sN:.1f} s"}}


def run_reference(args, ws_size, rank):
    """--impl reference: the oracle on every host core, each step a bounded
    sample of the workload (whole-T channel columns, one oracle call per
    core)."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    samples = [_sample(seed) for seed in range(4)]
    t = time.perf_counter()
    _oracle_fwd_bwd(samples[0])
    per_call = time.perf_counter() - t
    # each step: `reps` calls per core, about 2 s of work on every core
    reps = int(min(200, max(1, 2.0 / max(per_call, 1e-3))))

    def one_step():
        stop_calls = reps * cores
        done = [0]
        lock = threading.Lock()
        els = [0]

        def worker(w):
            while True:
                with lock:
                    if done[0] >= stop_calls:
                        return
                    i = done[0]
                    done[0] += 1
                e = _oracle_fwd_bwd(samples[i % len(samples)])
                with lock:
                    els[0] += e

        t0 = time.perf_counter()
        ths = [threading.Thread(target=worker, args=(w,)) for w in range(cores)]
        for th in ths:
            th.start()
        for th in ths:
            th.join()
        return els[0], time.perf_counter() - t0

    for _ in range(args.warmup):
        one_step()
    els, secs = 0, 0.0
    for _ in range(args.steps):
        e, s = one_step()
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
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"{reps * cores} oracle calls per step on {SAMPLE_COLS} "
                                   f"whole-T channel columns of {WORKLOAD}, {cores} threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
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
