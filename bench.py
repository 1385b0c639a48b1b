#!/usr/bin/env python3
"""Benchmark of the GB300 axis reductions.

One step = one pass of every reduction over the five synthetic workloads:

  full    2**20 fp32 U[-1,1)               sum, max, min
  rows    65536 x 1024 fp32 N(0,1)         sum, max, min, sum with accum
  full    2**30 fp32 N(0,1) (4 GiB)        sum, max, min
  colprod 4096 x 16384 fp32 U[.999,1.001]  and 64 x 65536 int32 {+-1,+-2,+-3}
  ragged  2**22 rows of 8..40 fp32 U[-4,4) sum, max, min

The ops run interleaved (every buffer is re-read only after at least 4 GiB of
other reads, so each op sees cold L2).  ``value`` is the algorithmic bytes of
a step (each input read once, each output written once) over the device time
of the step, in GB/s, summed over ranks (weak scaling: every rank runs the
whole workload on its own GPU).  Per-op times, the roofline of the dominant
kernel (the 4 GiB full reduction), an end-to-end figure through host buffers,
the grid-stage comparison of the full reduction, and the CPU oracle timed on
a sample of the same workload go into the same JSON line.

``--impl reference`` times the CPU oracle alone on the host (no GPU), one
bounded sample of the workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s (and % of ~8 TB/s) for full/row sum-max-min and col-prod"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = ("all five reduction workloads, one pass of every op: full 2^20 + full 2^30 (sum/max/min), "
            "rows 65536x1024 (sum/max/min + sum accum), colprod f32 4096x16384 + i32 64x65536, "
            "ragged 2^22 rows of 8..40 (sum/max/min)")
DOMINANT = "seg_kernel (red_full, 2^30 fp32 sum/max/min)"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = [os.path.join(ROOT, "int_tensor_reductions_gb300", "csrc", f)
                  for f in ("red_full.cu", "red_prims.cuh")] + [os.path.join(ROOT, "include", "red_device.cuh")]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stage-compare", action="store_true")
    ap.add_argument("--no-supplementary", action="store_true",
                    help="skip the 1 GiB row and column-product cases that grade the >= 1 GiB bars")
    ap.add_argument("--only", default="",
                    help="comma-separated op families to run (full1, full3, rows2, ragged5, colprod4a, "
                         "colprod4b); for profiling: the line is then not the benchmark's metric")
    ap.add_argument("--scale", type=float, default=1.0,
                    help="fraction of every workload's size (rows / elements); for profiling")
    ap.add_argument("--sweep", action="store_true",
                    help="print per-call GB/s of every entry point over a range of shapes (one JSON line "
                         "per case, CUDA-graph replays), then exit; not the benchmark's metric")
    ap.add_argument("--case", default="", choices=[""] + sorted(CASES),
                    help="run one extra library case (not the step) --steps times after --warmup, for profiling")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def sha_of(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


def traffic_per_launch():
    """DRAM bytes per launch of the dominant kernel from the last ncu capture,
    or None when none was taken of the kernel as it is now."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("sources_sha256") != sha_of(KERNEL_SOURCES):
        return None
    return t.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.window = None
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), line.strip()))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return self.summarize(self.samples, self.window)

    @classmethod
    def summarize(cls, samples, window):
        """Median SM clock, max clock and active throttle reasons of the
        (time, nvidia-smi csv line) samples inside window (t0, t1), or of the
        sample nearest its middle if none falls inside; None without samples."""
        rows = []
        for t, line in samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                rows.append((t, float(parts[0]), float(parts[1]), parts[4:]))
            except ValueError:
                continue
        if not rows:
            return None
        t0, t1 = window or (rows[0][0], rows[-1][0])
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05] or \
            [min(rows, key=lambda r: abs(r[0] - (t0 + t1) / 2))]
        reasons = sorted({name for r in inside for name, v in zip(cls.NAMES, r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The largest x over all ranks (x itself without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0])


def job_gbs(world: int, step_bytes: int, steps: int, max_ms: float) -> float:
    """Whole-job GB/s: every rank processed steps x step_bytes in at most max_ms."""
    return world * step_bytes * steps / (max_ms * 1e-3) / 1e9


# ----------------------------------------------------- single extra cases

def _case_inputs(name, dev):
    """(callable, algorithmic bytes per call) of one extra library case."""
    import torch
    import int_tensor_reductions_gb300 as itr
    from int_tensor_reductions_gb300 import synth
    if name == "stats_full_2p28":
        x = synth.normal((1 << 28,), 2, dev)
        o = torch.empty(4, device=dev)
        return (lambda: itr.red_full_stats(x, o)), 4 * x.numel() + 16
    if name == "stats_rows_65536x1024":
        x, _ = synth.cfg2(dev)
        o = torch.empty((x.shape[0], 4), device=dev)
        return (lambda: itr.red_rows_stats(x, o)), 4 * x.numel() + 16 * x.shape[0]
    if name == "thread_rows_2p22x32":
        x = synth.normal((1 << 22, 32), 3, dev)
        o = torch.empty(1 << 22, device=dev)
        return (lambda: itr.red_rows_thread("sum", x, out=o)), 4 * x.numel() + 4 * x.shape[0]
    if name == "cols_f16_prod_4096x16384":
        x = synth.col_input("prod", "f16", (4096, 16384), 11, dev)
        o = torch.empty(16384, dtype=x.dtype, device=dev)
        return (lambda: itr.red_cols("prod", x, o)), 2 * x.numel() + 2 * 16384
    if name == "typed_full_f16_max_2p29":
        x = synth.col_input("max", "f16", (1 << 29,), 12, dev)
        o = torch.empty(1, dtype=x.dtype, device=dev)
        return (lambda: itr.red_full_typed("max", x, o)), 2 * x.numel() + 2
    if name == "typed_rows_bf16_max_65536x2048":
        x = synth.col_input("max", "bf16", (65536, 2048), 12, dev)
        o = torch.empty(65536, dtype=x.dtype, device=dev)
        return (lambda: itr.red_rows_typed("max", x, out=o)), 2 * x.numel() + 2 * 65536
    if name == "typed_rows_u16_max_2p24x8":
        x = synth.col_input("max", "u16", (1 << 24, 8), 13, dev)
        o = torch.empty(1 << 24, dtype=x.dtype, device=dev)
        return (lambda: itr.red_rows_typed("max", x, out=o, dtype="u16")), 2 * x.numel() + 2 * (1 << 24)
    if name == "cols_bf16_sum_131072x1024":
        x = synth.col_input("sum", "bf16", (131072, 1024), 14, dev)
        o = torch.empty(1024, dtype=x.dtype, device=dev)
        return (lambda: itr.red_cols("sum", x, o)), 2 * x.numel() + 2 * 1024
    if name == "rows_262144x1024":
        x = synth.normal((262144, 1024), 7, dev)
        o = torch.empty(262144, device=dev)
        return (lambda: itr.red_rows("sum", x, out=o)), 4 * x.numel() + 4 * 262144
    if name == "colprod_16384x16384":
        x = synth.uniform((16384, 16384), 0.999, 1.001, 8, dev)
        o = torch.empty(16384, device=dev)
        return (lambda: itr.red_colprod(x, o)), 4 * x.numel() + 4 * 16384
    if name == "ragged_short_2p25":
        off = synth.ragged_offsets(1 << 25, 2, 6, 15, dev)
        nnz = int(off[-1].item())
        x = synth.uniform((nnz,), -1.0, 1.0, 16, dev)
        o = torch.empty(1 << 25, device=dev)
        return (lambda: itr.red_rows_ragged("sum", x, off, out=o)), 4 * nnz + 8 * ((1 << 25) + 1) + 4 * (1 << 25)
    raise KeyError(name)


CASES = ("stats_full_2p28", "stats_rows_65536x1024", "thread_rows_2p22x32", "cols_f16_prod_4096x16384",
         "typed_full_f16_max_2p29", "typed_rows_bf16_max_65536x2048", "typed_rows_u16_max_2p24x8",
         "cols_bf16_sum_131072x1024", "ragged_short_2p25", "rows_262144x1024", "colprod_16384x16384")


def run_case(args):
    """One extra case, --warmup untimed then --steps timed calls (CUDA events);
    prints one JSON line.  Used for profiling single kernels."""
    import torch
    from int_tensor_reductions_gb300 import _build
    _build.build_lib()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    fn, nbytes = _case_inputs(args.case, dev)
    for _ in range(max(1, args.warmup)):
        fn()
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    print(json.dumps({"case": args.case, "ms": round(ms, 5), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                      "bytes_per_call": nbytes}), flush=True)
    return 0


# ------------------------------------------------------------ the workload

class Workload:
    """Device inputs and outputs of one step and the ops in step order."""

    def __init__(self, device, frac=1.0, host_only=False, kinds=None):
        import torch
        from int_tensor_reductions_gb300 import synth
        self.torch = torch
        gen_dev = "cpu" if host_only else device

        def n_of(n, kind):
            # workloads left out by `kinds` get token-sized inputs
            f = frac if (not kinds or kind in kinds) else 1.0 / 65536
            return max(8, int(n * f))

        self.x1 = synth.cfg1(gen_dev, n=n_of(synth.CFG1_N, "full1"))
        self.x2, self.dst2 = synth.cfg2(gen_dev, rows=n_of(synth.CFG2_ROWS, "rows2"), length=synth.CFG2_LEN)
        self.x3 = synth.cfg3(gen_dev, n=n_of(synth.CFG3_N, "full3"))
        self.x4a = synth.cfg4a(gen_dev, R=n_of(synth.CFG4A_R, "colprod4a"), C=synth.CFG4A_C)
        self.x4b = synth.cfg4b(gen_dev, R=n_of(synth.CFG4B_R, "colprod4b"), C=synth.CFG4B_C)
        self.x5, self.off5 = synth.cfg5(gen_dev, rows=n_of(synth.CFG5_ROWS, "ragged5"))
        self.inputs = [self.x1, self.x2, self.dst2, self.x3, self.x4a, self.x4b, self.x5, self.off5]
        r2, l2 = self.x2.shape
        n5 = self.off5.numel() - 1
        nnz5 = self.x5.numel()
        self.bytes_of = {
            "full1": 4 * self.x1.numel() + 4,
            "full3": 4 * self.x3.numel() + 4,
            "rows2": 4 * r2 * l2 + 4 * r2,
            "rows2_accum": 4 * r2 * l2 + 8 * r2,
            "colprod4a": 4 * self.x4a.numel() + 4 * self.x4a.shape[1],
            "colprod4b": 4 * self.x4b.numel() + 4 * self.x4b.shape[1],
            "ragged5": 4 * nnz5 + 8 * (n5 + 1) + 4 * n5,
        }
        # input elements each op reduces (for elements per second)
        self.elems_of = {
            "full1": self.x1.numel(), "full3": self.x3.numel(), "rows2": r2 * l2, "rows2_accum": r2 * l2,
            "colprod4a": self.x4a.numel(), "colprod4b": self.x4b.numel(), "ragged5": nnz5,
        }
        # step order: interleaved so that no buffer is re-read while hot
        self.plan = [
            ("full1 sum", "full1"), ("full3 sum", "full3"), ("rows2 sum", "rows2"), ("ragged5 sum", "ragged5"),
            ("colprod4a f32", "colprod4a"),
            ("full1 max", "full1"), ("full3 max", "full3"), ("rows2 max", "rows2"), ("ragged5 max", "ragged5"),
            ("colprod4b i32", "colprod4b"),
            ("full1 min", "full1"), ("full3 min", "full3"), ("rows2 min", "rows2"), ("ragged5 min", "ragged5"),
            ("rows2 sum accum", "rows2_accum"),
        ]
        self.step_bytes = sum(self.bytes_of[k] for _, k in self.plan)
        if not host_only:
            t = torch
            self.o1 = {op: t.empty(1, device=device) for op in ("sum", "max", "min")}
            self.o3 = {op: t.empty(1, device=device) for op in ("sum", "max", "min")}
            self.o2 = {op: t.empty(r2, device=device) for op in ("sum", "max", "min")}
            self.o2acc = self.dst2.clone()
            self.o4a = t.empty(self.x4a.shape[1], device=device)
            self.o4b = t.empty(self.x4b.shape[1], dtype=t.int32, device=device)
            self.o5 = {op: t.empty(n5, device=device) for op in ("sum", "max", "min")}
            self.outputs = list(self.o1.values()) + list(self.o3.values()) + list(self.o2.values()) + \
                [self.o2acc, self.o4a, self.o4b] + list(self.o5.values())

    def gpu_call(self, name):
        import int_tensor_reductions_gb300 as itr
        kind, op = name.split(" ")[0], name.split(" ")[1]
        if kind == "full1":
            return lambda: itr.red_full(op, self.x1, self.o1[op])
        if kind == "full3":
            return lambda: itr.red_full(op, self.x3, self.o3[op])
        if kind == "rows2" and name.endswith("accum"):
            return lambda: itr.red_rows("sum", self.x2, accum=True, out=self.o2acc)
        if kind == "rows2":
            return lambda: itr.red_rows(op, self.x2, out=self.o2[op])
        if kind == "ragged5":
            return lambda: itr.red_rows_ragged(op, self.x5, self.off5, out=self.o5[op])
        if kind == "colprod4a":
            return lambda: itr.red_colprod(self.x4a, self.o4a)
        if kind == "colprod4b":
            return lambda: itr.red_colprod(self.x4b, self.o4b)
        raise KeyError(name)


def oracle_step(w: Workload, host):
    """One pass of every op through the CPU oracle on host arrays; returns
    the seconds spent inside the oracle calls."""
    import oracle
    x1, x2, dst2, x3, x4a, x4b, x5, off5 = host
    r2, l2 = x2.shape
    R4a, C4a = x4a.shape
    R4b, C4b = x4b.shape
    t = 0.0
    for name, _ in w.plan:
        kind, op = name.split(" ")[0], name.split(" ")[1]
        t0 = time.perf_counter()
        if kind == "full1":
            oracle.full(op, x1)
        elif kind == "full3":
            oracle.full(op, x3)
        elif kind == "rows2" and name.endswith("accum"):
            oracle.rows("sum", x2, r2, l2, True, dst2)
        elif kind == "rows2":
            oracle.rows(op, x2, r2, l2)
        elif kind == "ragged5":
            oracle.ragged(op, x5, off5)
        elif kind == "colprod4a":
            oracle.colprod_f32(x4a, R4a, C4a)
        else:
            oracle.colprod_i32(x4b, R4b, C4b)
        t += time.perf_counter() - t0
    return t


# ------------------------------------------------------------- reference

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np  # noqa: F401
    # Size each step's sample so that warm-up plus timed steps stay near
    # two minutes of single-thread oracle time (calibrated on a small probe).
    probe = Workload(None, frac=1.0 / 256, host_only=True)
    host = [t.numpy() for t in probe.inputs]
    t_probe = max(oracle_step(probe, host), 1e-6)
    full_est = t_probe * 256
    budget = 120.0 / max(1, args.steps + args.warmup)
    frac = min(1.0, max(1.0 / 256, budget / full_est))
    w = Workload(None, frac=frac, host_only=True)
    host = [t.numpy() for t in w.inputs]
    for _ in range(args.warmup):
        oracle_step(w, host)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, host)
    dt = time.perf_counter() - t0
    value = w.step_bytes * args.steps / dt / 1e9
    sample = f"{frac:.4g} of every workload (leading rows / elements), {w.step_bytes} bytes per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32/i32",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ ours

def run_ours(args):
    import torch
    import int_tensor_reductions_gb300 as itr
    from int_tensor_reductions_gb300 import _build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device; this library has no CPU path")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.build_lib()
    stream = torch.cuda.current_stream(dev)

    only = [k for k in args.only.split(",") if k]
    w = Workload(dev, frac=args.scale, kinds=only or None)
    partial = bool(only) or args.scale != 1.0
    if only:
        w.plan = [(name, key) for name, key in w.plan if name.split(" ")[0] in only]
        w.step_bytes = sum(w.bytes_of[k] for _, k in w.plan)
    if partial:
        args.no_e2e = args.no_cpu_baseline = args.no_supplementary = True
        args.no_stage_compare = args.no_stage_compare or "full3" not in (only or ["full3"])
    calls = [(name, key, w.gpu_call(name)) for name, key in w.plan]
    torch.cuda.synchronize()

    def step():
        for _, _, fn in calls:
            fn()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    # (1) eager pass (host-launched calls, no graph): its step time is
    # reported beside the graph's
    K = args.steps
    KE = min(K, 20)
    torch.cuda.synchronize()
    e_begin, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_begin.record(stream)
    for k in range(KE):
        step()
    e_end.record(stream)
    torch.cuda.synchronize()
    eager_ms = e_begin.elapsed_time(e_end) / KE

    # (2) the timed region: the step captured once as a CUDA graph (the same
    # library calls, no host launch gaps between them) and replayed K times
    graph = torch.cuda.CUDAGraph()
    launches0 = itr.red_launch_count()
    with torch.cuda.graph(graph):
        step()
    kernels_per_step = itr.red_launch_count() - launches0
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    if vis and vis.split(",")[0].strip().isdigit():
        gpu_index = int(vis.split(",")[local].strip())
    sampler = ClockSampler(gpu_index)
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    h0 = time.monotonic()
    t_begin.record(stream)
    for _ in range(K):
        graph.replay()
    t_end.record(stream)
    torch.cuda.synchronize()
    h1 = time.monotonic()
    if dist:
        dist.barrier()
    launches = kernels_per_step * K
    sampler.mark(h0, h1)
    clocks = sampler.stop()
    total_ms = max_over_ranks(t_begin.elapsed_time(t_end), dist, dev)
    value = job_gbs(world, w.step_bytes, K, total_ms)
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks and "hbm_gbs" in peaks else FALLBACK_HBM_GBS
    peak_src = "measured" if peaks and "hbm_gbs" in peaks else "fallback"
    # (3) per-op device time from CUDA graphs (each op's calls back to back)
    per_op, ops_note = per_op_graphs(w, stream)
    dom = [per_op[n]["ms"] for n in ("full3 sum", "full3 max", "full3 min") if n in per_op]
    dom_ms = sum(dom) / len(dom) if dom else float("nan")
    achieved = w.bytes_of["full3"] / (dom_ms * 1e-3) / 1e9 if dom else None
    ops_sum = sum(v["ms"] for v in per_op.values())

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": round(total_ms / K, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32/i32", "data": "synthetic",
        "config": {
            "workload": WORKLOAD,
            "bytes_per_step": w.step_bytes,
            "l2": "inputs larger than L2 between reuses: ops interleaved so every buffer is re-read only "
                  "after >= 4 GiB of other reads (L2 is 126 MiB)",
            "full_grid_stage": {0: "auto: two-pass for sum, atomic for max/min", 1: "two-pass", 2: "last-block",
                                3: "atomic"}[itr.red_get_full_mode()],
            "parallelism": f"replicas x{world}",
        },
        "frac_of_nominal_8TBs": round(value / world / NOMINAL_HBM_GBS, 4),
        "gelem_s": round(world * sum(w.elems_of[k] for _, k in w.plan) * K / (total_ms * 1e-3) / 1e9, 2),
        "roofline": {
            "bound": "hbm", "kernel": DOMINANT, "achieved": achieved and round(achieved, 1), "peak": peak,
            "unit": "GB/s", "frac": achieved and round(achieved / peak, 4), "peak_source": peak_src,
            "frac_of_nominal_8TBs": achieved and round(achieved / NOMINAL_HBM_GBS, 4),
            "traffic": traffic_per_launch(), "algorithmic_bytes_per_launch": w.bytes_of["full3"],
        },
        "ops": per_op,
        "timing": {"timed_region": f"CUDA graph of one step ({kernels_per_step} library kernels) replayed "
                                   f"{K} times", "eager_ms_per_step": round(eager_ms, 5),
                   "ops_from": ops_note, "ops_sum_ms": round(ops_sum, 5),
                   "ops_sum_over_ms_per_step": round(ops_sum / (total_ms / K), 4)},
        "gpu_launches": int(launches),
        "partial": {"only": only, "scale": args.scale} if partial else None,
        "clocks": clocks,
    }

    if not args.no_stage_compare:
        result["full_grid_stage_compare"] = compare_stages(w, stream)

    if not args.no_supplementary:
        result["small_cold_warm"] = small_cold_warm(w, stream)
        result["fused_stats_2p30"] = fused_stats(w, stream, per_op)
        result["supplementary_1gib"] = supplementary(stream, dev, peak)
        result["column_ops"] = column_ops(stream, dev, peak)
        result["typed_ops"] = typed_ops(stream, dev, peak)

    if not args.no_e2e:
        result["e2e"] = run_e2e(w, calls, stream, args.e2e_steps, world, dist, dev)

    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w)

    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def per_op_graphs(w, stream, calls_per_replay=16, replays=8):
    """Device time per call of every op of the step, each timed alone: one
    CUDA graph per op holding at least ``calls_per_replay`` back-to-back calls
    over copies of that op's inputs (so that every call reads its input cold:
    the copies together exceed three times the L2; a replay calls every copy
    once), after one warm-up replay ``replays`` replays queued back to back,
    each between two events on the launching stream.  Graph replay leaves no
    host launch gap, and programmatic dependent launch overlaps each call's
    launch with its predecessor's drain, as in the timed region.  Per op: the
    median and the best replay's time per call, GB/s of algorithmic bytes and
    input elements per second from the median."""
    import statistics
    import torch
    import int_tensor_reductions_gb300 as itr
    l2 = torch.cuda.get_device_properties(stream.device).L2_cache_size

    def copies(t):
        n = max(1, -(-3 * l2 // max(1, t.numel() * t.element_size())))
        return [t] + [t.clone() for _ in range(n - 1)]

    x1s, x2s, x4as, x4bs = copies(w.x1), copies(w.x2), copies(w.x4a), copies(w.x4b)
    x3s, x5s = copies(w.x3), copies(w.x5)

    def fns(name):
        kind, op = name.split(" ")[0], name.split(" ")[1]
        if kind == "full1":
            return [lambda x=x: itr.red_full(op, x, w.o1[op]) for x in x1s]
        if kind == "full3":
            return [lambda x=x: itr.red_full(op, x, w.o3[op]) for x in x3s]
        if kind == "rows2" and name.endswith("accum"):
            return [lambda x=x: itr.red_rows("sum", x, accum=True, out=w.o2acc) for x in x2s]
        if kind == "rows2":
            return [lambda x=x: itr.red_rows(op, x, out=w.o2[op]) for x in x2s]
        if kind == "ragged5":
            return [lambda x=x: itr.red_rows_ragged(op, x, w.off5, out=w.o5[op]) for x in x5s]
        if kind == "colprod4a":
            return [lambda x=x: itr.red_colprod(x, w.o4a) for x in x4as]
        return [lambda x=x: itr.red_colprod(x, w.o4b) for x in x4bs]

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(replays + 1)]
    per_op = {}
    for name, key in w.plan:
        f = fns(name)
        for fn in f:
            fn()
        torch.cuda.synchronize()
        ncalls = max(calls_per_replay, len(f))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for k in range(ncalls):
                f[k % len(f)]()
        g.replay()
        torch.cuda.synchronize()
        ev[0].record(stream)
        for k in range(replays):
            g.replay()
            ev[k + 1].record(stream)
        torch.cuda.synchronize()
        per_call = [ev[k].elapsed_time(ev[k + 1]) / ncalls for k in range(replays)]
        ms, best = statistics.median(per_call), min(per_call)
        per_op[name] = {"ms": round(ms, 5), "gbs": round(w.bytes_of[key] / (ms * 1e-3) / 1e9, 1),
                        "best_ms": round(best, 5), "gelem_s": round(w.elems_of[key] / (ms * 1e-3) / 1e9, 2)}
        del g
    del x1s, x2s, x4as, x4bs, x3s, x5s
    torch.cuda.empty_cache()
    note = (f"graph-timed per op: at least {calls_per_replay} back-to-back calls per CUDA graph over copies of the "
            f"op's inputs (each call reads cold); median (ms, gbs, gelem_s) and best of {replays} replays")
    return per_op, note


def compare_stages(w, stream, reps=10):
    """GB/s of the 4 GiB full reduction under each grid stage."""
    import torch
    import int_tensor_reductions_gb300 as itr
    keep = itr.red_get_full_mode()
    out = {}
    for mode, label in ((itr.RED_MODE_TWO_PASS, "two-pass"), (itr.RED_MODE_LAST_BLOCK, "last-block"),
                        (itr.RED_MODE_ATOMIC, "atomic")):
        itr.red_set_full_mode(mode)
        res = {}
        for op in ("sum", "max", "min"):
            for _ in range(2):
                itr.red_full(op, w.x3, w.o3[op])
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(reps):
                itr.red_full(op, w.x3, w.o3[op])
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / reps
            res[op] = round(w.bytes_of["full3"] / (ms * 1e-3) / 1e9, 1)
        out[label] = res
    itr.red_set_full_mode(keep)
    return {"unit": "GB/s", "note": "2^30 fp32, back-to-back calls (4 GiB > L2)", **out}


def fused_stats(w, stream, per_op, reps=10):
    """red_full_stats (sum, max, min, sum|x| from one read) on the 2^30 vector,
    against the three separate red_full calls of the step."""
    import torch
    import int_tensor_reductions_gb300 as itr
    out = torch.empty(4, device=w.x3.device)
    for _ in range(2):
        itr.red_full_stats(w.x3, out)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        itr.red_full_stats(w.x3, out)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    sep = sum(per_op[f"full3 {op}"]["ms"] for op in ("sum", "max", "min") if f"full3 {op}" in per_op)
    res = {"ms": round(ms, 4), "gbs": round(w.bytes_of["full3"] / (ms * 1e-3) / 1e9, 1),
           "separate_sum_max_min_ms": round(sep, 4), "speedup_vs_separate": round(sep / ms, 3) if sep else None}
    # per-row statistics of the 65536 x 1024 rows, against the three row ops
    r2, l2 = w.x2.shape
    ro = torch.empty((r2, 4), device=w.x2.device)
    for _ in range(2):
        itr.red_rows_stats(w.x2, ro)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        itr.red_rows_stats(w.x2, ro)
    e1.record(stream)
    torch.cuda.synchronize()
    rms = e0.elapsed_time(e1) / reps
    rsep = sum(per_op[f"rows2 {op}"]["ms"] for op in ("sum", "max", "min") if f"rows2 {op}" in per_op)
    res["rows_65536x1024"] = {"ms": round(rms, 4), "gbs": round((4 * r2 * l2 + 16 * r2) / (rms * 1e-3) / 1e9, 1),
                              "separate_sum_max_min_ms": round(rsep, 4),
                              "speedup_vs_separate": round(rsep / rms, 3) if rsep else None}
    return res


def small_cold_warm(w, stream, calls=20, reps=50):
    """The two L2-sized workloads (the 2**20 vector, 4 MiB, and the 64 x 65536
    int32 column product, 16 MiB), per call.  Single calls are too short for
    CUDA events (their timestamps step by ~2 us), so the calls are captured
    in CUDA graphs and each graph is replayed ``reps`` times between two
    events: warm = ``calls`` back-to-back calls (the input stays in L2) per
    replay; cold = ``calls`` pairs of (write twice the L2 size, call) minus
    the same graph without the calls."""
    import torch
    l2 = torch.cuda.get_device_properties(stream.device).L2_cache_size
    scratch = torch.empty(2 * l2 // 4 + 1, dtype=torch.float32, device=stream.device)

    def per_replay(body):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            body()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps  # us

    res = {"unit": "us", "note": f"per call, from CUDA-graph replays ({calls} calls per graph, {reps} replays); "
                                 f"cold: {2 * l2 >> 20} MiB written before each call, that write's own time "
                                 "subtracted"}
    flushes = per_replay(lambda: [scratch.fill_(1.0) for _ in range(calls)])
    for name in ("full1 sum", "full1 max", "full1 min", "colprod4b i32"):
        if name not in dict(w.plan):
            continue
        fn = w.gpu_call(name)
        nbytes = w.bytes_of[dict(w.plan)[name]]
        fn()
        torch.cuda.synchronize()
        warm = per_replay(lambda: [fn() for _ in range(calls)]) / calls
        both = per_replay(lambda: [(scratch.fill_(1.0), fn()) for _ in range(calls)])
        cold = (both - flushes) / calls
        res[name] = {"warm_us": round(warm, 2), "cold_us": round(cold, 2),
                     "warm_gbs": round(nbytes / (warm * 1e-6) / 1e9, 1),
                     "cold_gbs": round(nbytes / (cold * 1e-6) / 1e9, 1)}
    del scratch
    torch.cuda.empty_cache()
    return res


def graph_ms_per_call(fn, stream, calls=10, replays=5):
    """Device time per call of ``calls`` back-to-back calls captured in one
    CUDA graph and replayed ``replays`` times between two events, so that the
    host's launch rate never leaves the GPU idle between short calls."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(calls):
            fn()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(replays):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (replays * calls)
    del g
    return ms


def supplementary(stream, dev, peak, reps=10):
    """The >= 1 GiB cases that grade the bandwidth bars of the row reductions
    and the column products (not part of the step): 262144 x 1024 fp32 rows
    (sum, max) and a 16384 x 16384 fp32 column product.  Back-to-back calls on
    1 GiB inputs (> L2)."""
    import torch
    import int_tensor_reductions_gb300 as itr
    from int_tensor_reductions_gb300 import synth
    out = {"unit": "GB/s", "note": "1 GiB inputs, back-to-back calls replayed from a CUDA graph, not part of the step"}

    def timed(fn):
        return graph_ms_per_call(fn, stream, calls=reps)

    x = synth.normal((262144, 1024), 7, dev)
    o = torch.empty(262144, device=dev)
    nbytes = 4 * x.numel() + 4 * 262144
    for op in ("sum", "max"):
        ms = timed(lambda: itr.red_rows(op, x, out=o))
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[f"rows 262144x1024 {op}"] = {"gbs": round(gbs, 1), "frac_of_nominal_8TBs": round(gbs / NOMINAL_HBM_GBS, 4),
                                         "frac_of_peak": round(gbs / peak, 4)}
    del x, o
    x = synth.uniform((16384, 16384), 0.999, 1.001, 8, dev)
    o = torch.empty(16384, device=dev)
    nbytes = 4 * x.numel() + 4 * 16384
    ms = timed(lambda: itr.red_colprod(x, o))
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["colprod f32 16384x16384"] = {"gbs": round(gbs, 1), "frac_of_nominal_8TBs": round(gbs / NOMINAL_HBM_GBS, 4),
                                      "frac_of_peak": round(gbs / peak, 4)}
    del x, o
    torch.cuda.empty_cache()
    return out


def column_ops(stream, dev, peak, reps=10):
    """Column reductions of the other element types and operators (TCOLPROD's
    siblings), each on an input larger than L2: GB/s of algorithmic bytes."""
    import torch
    import int_tensor_reductions_gb300 as itr
    from int_tensor_reductions_gb300 import synth
    res = {"unit": "GB/s", "note": "back-to-back calls replayed from a CUDA graph, inputs > L2 except the 8 MiB "
                                   "int16 case (L2-resident between calls)"}
    for op, dtype, R, C in (("sum", "f32", 4096, 16384), ("prod", "f16", 4096, 16384), ("sum", "bf16", 8192, 16384),
                            ("max", "u32", 4096, 16384), ("prod", "i16", 64, 65536)):
        x = synth.col_input(op, dtype, (R, C), 11, dev)
        o = torch.empty(C, dtype=x.dtype, device=dev)
        ms = graph_ms_per_call(lambda: itr.red_cols(op, x, o, dtype=dtype), stream, calls=reps)
        nbytes = x.numel() * x.element_size() + C * x.element_size()
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[f"{op} {dtype} {R}x{C}"] = {"us": round(ms * 1e3, 1), "gbs": round(gbs, 1),
                                       "frac_of_peak": round(gbs / peak, 4)}
        del x, o
    torch.cuda.empty_cache()
    return res


def typed_ops(stream, dev, peak, reps=10):
    """Full and row reductions of other element types (red_full_typed,
    red_rows_typed) on inputs larger than L2: GB/s of algorithmic bytes; the
    fp32 rows of the same shape through red_rows, timed the same way."""
    import torch
    import int_tensor_reductions_gb300 as itr
    from int_tensor_reductions_gb300 import synth
    res = {"unit": "GB/s", "note": "back-to-back calls replayed from a CUDA graph, inputs > L2"}
    cases = (("full", "sum", "i32", (1 << 28,)), ("full", "max", "f16", (1 << 29,)),
             ("rows", "sum", "i32", (65536, 1024)), ("rows", "sum", "f32", (65536, 1024)),
             ("rows", "max", "bf16", (65536, 2048)))
    for kind, op, dtype, shape in cases:
        x = synth.col_input(op, dtype, shape, 12, dev)
        if kind == "rows" and dtype == "f32":
            o = torch.empty(shape[0], dtype=x.dtype, device=dev)
            fn = lambda: itr.red_rows(op, x, out=o)  # noqa: E731
        elif kind == "full":
            o = torch.empty(1, dtype=x.dtype, device=dev)
            fn = lambda: itr.red_full_typed(op, x, o, dtype=dtype)  # noqa: E731
        else:
            o = torch.empty(shape[0], dtype=x.dtype, device=dev)
            fn = lambda: itr.red_rows_typed(op, x, out=o, dtype=dtype)  # noqa: E731
        ms = graph_ms_per_call(fn, stream, calls=reps)
        nbytes = (x.numel() + o.numel()) * x.element_size()
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[f"{kind} {op} {dtype} {'x'.join(map(str, shape))}"] = {"us": round(ms * 1e3, 1), "gbs": round(gbs, 1),
                                                                   "frac_of_peak": round(gbs / peak, 4)}
        del x, o
    torch.cuda.empty_cache()
    return res


def run_e2e(w, calls, stream, steps, world, dist, dev):
    """The same step through the public API from pinned host buffers: every
    step copies its inputs host->device and its results device->host.

    The host->device copies run on a second stream and each workload's ops
    start as soon as its own inputs have landed, so the reductions overlap the
    remaining copies (the host link, not the GPU, bounds this figure: ~211
    GB/s host->device on this machine).  The ragged rows go first (their 48 MB
    of results then travel back on a third stream while the other inputs are
    still arriving), the 4 GiB vector second (its reductions run while the
    rest is copied), the small inputs last.  Each workload's results are
    copied back as soon as its ops are done; the step ends when every copy
    has landed."""
    import torch
    host_in = [t.cpu().pin_memory() for t in w.inputs]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in w.outputs]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    copy_stream = torch.cuda.Stream(device=dev)
    back_stream = torch.cuda.Stream(device=dev)
    # inputs each op family reads (indices into w.inputs) and the outputs it
    # writes (indices into w.outputs)
    needs = {"full1": [0], "rows2": [1, 2], "full3": [3], "colprod4a": [4], "colprod4b": [5], "ragged5": [6, 7]}
    writes = {"full1": [0, 1, 2], "full3": [3, 4, 5], "rows2": [6, 7, 8, 9], "colprod4a": [10], "colprod4b": [11],
              "ragged5": [12, 13, 14]}
    order = [6, 7, 3, 1, 2, 4, 0, 5]  # ragged rows, then the 4 GiB vector, then the rest
    fam_order = ["ragged5", "full3", "rows2", "colprod4a", "full1", "colprod4b"]

    def step():
        start = torch.cuda.Event()
        start.record(stream)
        copy_stream.wait_event(start)
        landed = {}
        with torch.cuda.stream(copy_stream):
            for i in order:
                w.inputs[i].copy_(host_in[i], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_stream)
                landed[i] = ev
        for fam in fam_order:
            for i in needs[fam]:
                stream.wait_event(landed[i])
            for name, _, fn in calls:
                if name.split(" ")[0] == fam:
                    fn()
            done = torch.cuda.Event()
            done.record(stream)
            back_stream.wait_event(done)
            with torch.cuda.stream(back_stream):
                for j in writes[fam]:
                    host_out[j].copy_(w.outputs[j], non_blocking=True)
        stream.wait_stream(back_stream)

    step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    value = job_gbs(world, w.step_bytes, steps, ms)
    return {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "ms_per_step": round(ms / steps, 3),
            "h2d_gbs_seen": round(h2d / (ms / steps * 1e-3) / 1e9, 1)}


def cpu_baseline(w, min_seconds=10.0):
    """The oracle, single-threaded, over whole passes of the same workload
    (the same input bits, copied to the host), repeated until at least
    ``min_seconds`` of oracle time have accumulated."""
    host = [t.cpu().numpy() for t in w.inputs]
    secs, steps = 0.0, 0
    while steps == 0 or secs < min_seconds:
        secs += oracle_step(w, host)
        steps += 1
    return {"value": round(steps * w.step_bytes / secs / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{steps} full steps (all 15 ops on the full-size inputs), single thread",
            "seconds": round(secs, 2), "host_cpus": os.cpu_count()}


def run_sweep(args):
    """Per-call device GB/s (algorithmic bytes over graph-replayed time) of
    the entry points across shapes, from L2-sized to several GiB."""
    import torch
    import int_tensor_reductions_gb300 as itr
    from int_tensor_reductions_gb300 import _build, synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _build.build_lib()
    stream = torch.cuda.current_stream(dev)

    def emit(kind, shape, fn, nbytes):
        ms = graph_ms_per_call(fn, stream, calls=5, replays=4)
        print(json.dumps({"sweep": kind, "shape": shape, "us": round(ms * 1e3, 2),
                          "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}), flush=True)

    for n in (1 << 16, 1 << 20, 1 << 24, 1 << 28, 1 << 30, (1 << 31) + 3):
        x = synth.uniform((n,), -1.0, 1.0, 1, dev)
        o = torch.empty(1, device=dev)
        for op in ("sum", "max"):
            emit(f"red_full {op}", [n], lambda: itr.red_full(op, x, o), 4 * n + 4)
        del x, o
        torch.cuda.empty_cache()
    for rows, length in ((1 << 23, 16), (1 << 21, 64), (1 << 19, 256), (1 << 18, 1024), (1 << 12, 1 << 16),
                         (16, 1 << 24), (3, 1 << 28)):
        x = synth.uniform((rows, length), -1.0, 1.0, 2, dev)
        o = torch.empty(rows, device=dev)
        emit("red_rows sum", [rows, length], lambda: itr.red_rows("sum", x, out=o), 4 * rows * length + 4 * rows)
        del x, o
        torch.cuda.empty_cache()
    for mean in (4, 8, 24, 100, 1000):
        rows = (1 << 27) // mean
        off = synth.ragged_offsets(rows, max(1, mean // 2), mean + mean // 2, 3, dev)
        nnz = int(off[-1].item())
        x = synth.uniform((nnz,), -1.0, 1.0, 4, dev)
        o = torch.empty(rows, device=dev)
        emit("red_rows_ragged sum", [rows, f"lengths {max(1, mean // 2)}..{mean + mean // 2}"],
             lambda: itr.red_rows_ragged("sum", x, off, out=o), 4 * nnz + 8 * (rows + 1) + 4 * rows)
        del x, o, off
        torch.cuda.empty_cache()
    for R, C in ((1 << 20, 64), (1 << 16, 1024), (4096, 16384), (64, 1 << 20), (16384, 16384)):
        x = synth.uniform((R, C), -1.0, 1.0, 5, dev)
        o = torch.empty(C, device=dev)
        emit("red_cols sum", [R, C], lambda: itr.red_cols("sum", x, o), 4 * R * C + 4 * C)
        del x, o
        torch.cuda.empty_cache()
    for dtype, R, C in (("f16", 1 << 21, 64), ("f16", 8192, 16384), ("i16", 64, 1 << 21), ("bf16", 1 << 17, 1024)):
        x = synth.col_input("sum", dtype, (R, C), 6, dev)
        o = torch.empty(C, dtype=x.dtype, device=dev)
        emit(f"red_cols sum {dtype}", [R, C], lambda: itr.red_cols("sum", x, o, dtype=dtype),
             x.element_size() * (R * C + C))
        del x, o
        torch.cuda.empty_cache()
    for dtype, shape in (("f16", (1 << 28,)), ("i32", (1 << 27,)), ("bf16", (1 << 22, 64)), ("i32", (1 << 23, 16)),
                         ("f16", (4096, 1 << 16)), ("u16", (1 << 24, 8)), ("i32", (1 << 26, 2)),
                         ("u16", (1 << 27, 1)), ("bf16", (1 << 23, 16)), ("f32", (1 << 25, 4)),
                         ("bf16", (1 << 21, 128)), ("f32", (1 << 21, 64)), ("i32", (1 << 19, 256))):
        x = synth.col_input("max", dtype, shape, 7, dev)
        if len(shape) == 1:
            o = torch.empty(1, dtype=x.dtype, device=dev)
            emit(f"red_full_typed max {dtype}", list(shape), lambda: itr.red_full_typed("max", x, o, dtype=dtype),
                 x.element_size() * (x.numel() + 1))
        else:
            o = torch.empty(shape[0], dtype=x.dtype, device=dev)
            emit(f"red_rows_typed max {dtype}", list(shape), lambda: itr.red_rows_typed("max", x, out=o, dtype=dtype),
                 x.element_size() * (x.numel() + shape[0]))
        del x, o
        torch.cuda.empty_cache()
    x = synth.uniform((1 << 28,), -1.0, 1.0, 8, dev)
    o = torch.empty(4, device=dev)
    emit("red_full_stats", [1 << 28], lambda: itr.red_full_stats(x, o), 4 * (1 << 28) + 16)
    del x, o
    for rows, length in ((1 << 23, 16), (1 << 22, 32), (1 << 21, 64), (1 << 17, 1024)):
        x = synth.uniform((rows, length), -1.0, 1.0, 9, dev)
        o = torch.empty((rows, 4), device=dev)
        emit("red_rows_stats", [rows, length], lambda: itr.red_rows_stats(x, o), 4 * rows * length + 16 * rows)
        del x, o
        torch.cuda.empty_cache()
    return 0


def main():
    args = parse_args()
    if args.sweep:
        return run_sweep(args)
    if args.case:
        return run_case(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
