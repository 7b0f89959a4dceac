#!/usr/bin/env python3
"""Benchmark of the whole SpMV path on one GB300 (or N replicas).

One step = one pass of every stage of the path over one matrix already
resident in HBM:
  create (validation + row statistics + nnz-balanced CSR partition),
  convert to COO, ELL, HYB (automatic width) and JDS, select,
  and y <- A x + y once in each of CSR, COO, ELL, HYB and JDS, then destroy.
The metric counts the compulsory SpMV bytes of the five products:
  effective GB/s = 5 * (8*nnz + 12*rows + 4*cols) / step time,
  GFLOP/s        = 5 * 2*nnz / step time.
The timed steps carry no events between their calls. A separate pass of
the same steps (CALL_STEPS of them) with a CUDA event between every two calls
gives each stage's own time and GB/s (`calls`); those events add about 2 us
per call boundary, so the calls sum to a little more than the step. `roofline` reports the kernel with the largest share of the workload's
ncu launch list, timed by the events of the call that launches it alone,
with its per-launch DRAM traffic from the committed capture; it also names
the call with the largest share of the step and the fastest SpMV.
The e2e figure repeats the step through the same C ABI with the inputs in
pinned host memory: every step's host-to-device copy of the CSR arrays, x and
y0 and the device-to-host read of its five results are inside the timed
region; the copies of neighbouring steps overlap the compute on their own
streams (two device buffer sets).

The default workload is the largest of the five (the 27-point stencil on
160^3, 109.2M nonzeros). After the timed steps, `per_config` times every
format's SpMV alone on each of the five workloads with L2 flushed before every
run (the per-format protocol of --mode kernels, fewer reps), with the
selector's choice and the fastest format of each.

--impl reference times the CPU oracle (plain single-threaded C, fp64) on the
same workload and metric, on a bounded row sample per step.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload stencil27] [--no-e2e] [--no-cpu-baseline]
                       [--no-per-config]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = ("SpMV fp32 GFLOP/s & effective HBM GB/s (fraction of ~8 TB/s) per format, 1 GB300")
FORMATS = ("CSR", "COO", "ELL", "HYB", "JDS")
ALL_FORMATS = ("CSR", "COO", "ELL", "HYB", "JDS", "SELL", "XBLOCK")
DEFAULT_WORKLOAD = "stencil27"
CONFIG_ORDER = ("tiny_uniform", "laplace2d", "uniform_random", "skewed", "stencil27")
WORKLOAD_DESC = {
    "tiny_uniform": "uniform 4096x4096, 8 nnz/row (32,768 nnz)",
    "laplace2d": "2D 5-point Laplacian on 2048x2048, Dirichlet (4,194,304 rows, 20,963,328 nnz)",
    "uniform_random": "uniform random 1M x 1M, 5 nnz/row (5M nnz)",
    "skewed": "skewed 2M x 2M: rows of 10-20 nnz + 200 rows of 1000-5000 nnz",
    "stencil27": "3D 27-point stencil on 160^3, Dirichlet (4,096,000 rows, 109,215,352 nnz)",
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# nominal fp64 rate of a GB300 (the vector unit; no tensor fp64 path)
FP64_NOMINAL_GFLOPS = 1250.0

# Per workload, (call, kernel): the kernel with the largest share of the
# step's ncu launch list, and the library call whose CUDA-event time is that
# kernel's duration (the call launches that kernel alone). Workloads without
# a launch list take the single-kernel call with the longest event time.
# (The CSR -> ELL scatter stages rows of 24 to 32 entries through shared
# memory, k_csr_to_ell_staged, and reads narrower or wider ones directly,
# k_csr_to_ell.)
DOMINANT = {"laplace2d": ("convert_ell", "k_csr_to_ell"),
            "stencil27": ("convert_ell", "k_csr_to_ell_staged")}
# calls that launch exactly one kernel of the library (on every workload): the
# kernel's name, or the prefix of the names of its forms
SINGLE_KERNEL_CALLS = {"convert_ell": "k_csr_to_ell", "convert_coo": "k_expand_rows",
                       "spmv_CSR": "k_spmv_csr_wide", "spmv_COO": "k_spmv_coo",
                       "spmv_ELL": "k_spmv_ell"}


def traffic_record(workload, kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu capture
    (profiles/traffic_<workload>.json), or None when there is none for this
    workload or the kernel's source file changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("kernel") != kernel:
            return None
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != rec["source_sha256"]:
                return None
        return int(rec["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# steps of the per-call breakdown pass (events between the calls)
CALL_STEPS = 50


def compulsory_bytes(R, C, Z, vb=4):
    """Bytes an SpMV must move with vb-byte values: value + column per
    nonzero, rowPtrs and y read + write per row, x once."""
    return (vb + 4) * Z + (4 + 2 * vb) * R + vb * C


def call_bytes(name, R, C, Z, K_ell, K_hyb, hyb_tail):
    """Algorithmic bytes of each library call (what it must read and write)."""
    spmv = compulsory_bytes(R, C, Z)
    return {
        "create": 4 * (R + 1) + 4 * Z,
        "convert_coo": 4 * (R + 1) + 4 * Z,
        "convert_ell": 4 * (R + 1) + 8 * Z + 8 * R * K_ell + 4 * R,
        "convert_hyb": 4 * (R + 1) + 8 * Z + 8 * R * K_hyb + 4 * R + 12 * hyb_tail,
        "convert_jds": 4 * (R + 1) + 4 * R + 16 * Z,
        "spmv_CSR": spmv, "spmv_COO": spmv, "spmv_ELL": spmv, "spmv_HYB": spmv,
        "spmv_JDS": spmv,
    }[name]


def convert_bytes(fmt, R, C, Z, vb=4, width=0, tail=0, slots=0):
    """Algorithmic bytes of converting CSR to `fmt` with vb-byte values: what
    the conversion must read from CSR and write (width: ELL/HYB slots per
    row; tail: HYB's COO entries; slots: SELL/XBLOCK stored entries, padding
    included)."""
    rp = 4 * (R + 1)
    return {
        "COO": rp + 4 * Z,                                       # rowIdx written
        "ELL": rp + (4 + vb) * Z + (4 + vb) * R * width + 4 * R,  # + nnzPerRow
        "HYB": rp + (4 + vb) * Z + (4 + vb) * R * width + 4 * R + (8 + vb) * tail,
        "JDS": rp + 4 * R + 2 * (4 + vb) * Z,                     # perm, entries moved
        "SELL": rp + 4 * R + (4 + vb) * Z + (4 + vb) * slots,
        # columns read twice (count, scatter), values once; row, 16-bit
        # column and value written per slot
        "XBLOCK": 4 * Z + (4 + vb) * Z + (6 + vb) * slots,
    }[fmt]


class ClockSampler:
    """nvidia-smi clock/throttle samples every 100 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, rank, world, device, inp):
    import torch
    import spmv_sparse_storage_gb300 as sp

    R, C, Z = inp.num_rows, inp.num_cols, inp.nnz
    stream = torch.cuda.current_stream(device)
    def make_bufs():
        """One device-resident set of the step's inputs and outputs."""
        return {"rp": torch.from_numpy(inp.row_ptrs).to(device),
                "ci": torch.from_numpy(inp.col_idx).to(device),
                "va": torch.from_numpy(inp.value).to(device),
                "x": torch.from_numpy(inp.x).to(device),
                "ys": {f: torch.from_numpy(inp.y0).to(device) for f in FORMATS}}

    bufs0 = make_bufs()
    torch.cuda.synchronize(device)

    names = ["create", "convert_coo", "convert_ell", "convert_hyb", "convert_jds"] + \
            [f"spmv_{f}" for f in FORMATS]
    info = {}

    def step(bufs, events=None):
        ev = events
        i = 0
        rp, ci, va, x, ys = bufs["rp"], bufs["ci"], bufs["va"], bufs["x"], bufs["ys"]

        def mark():
            nonlocal i
            if ev is not None:
                ev[i].record(stream)
                i += 1

        mark()
        h = sp.spmv_create_csr(R, C, Z, rp, ci, va, stream)
        mark()
        sp.spmv_convert_coo(h, stream)
        mark()
        sp.spmv_convert_ell(h, stream)
        mark()
        sp.spmv_convert_hyb(h, 0, stream)
        mark()
        sp.spmv_convert_jds(h, stream)
        mark()
        fmt, width = sp.spmv_select(h)
        for f in FORMATS:
            sp.spmv_run(h, f, x, ys[f], stream)
            mark()
        if "auto" not in info:
            a = sp.spmv_export(h, "HYB")
            info.update(auto=fmt, hyb_width=width, hyb_tail=a["coo_nnz"],
                        ell_width=sp.spmv_export(h, "ELL")["width"])
        sp.spmv_destroy(h)

    for _ in range(args.warmup):
        step(bufs0)
    torch.cuda.synchronize(device)

    K = args.steps
    clocks = ClockSampler(device.index if device.index is not None else 0)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launches0 = sp.spmv_launch_count()
    t0.record(stream)
    for k in range(K):
        step(bufs0)
    t1.record(stream)
    torch.cuda.synchronize(device)
    launches = sp.spmv_launch_count() - launches0
    barrier(world)
    clk = clocks.stop() if rank == 0 else None
    elapsed_ms = t0.elapsed_time(t1)
    elapsed_ms = allreduce_max(elapsed_ms, world, device)

    # Per-call breakdown: a separate pass of the same steps with an event
    # between every two calls (the events themselves add about 2 us per call
    # boundary, so the step above is timed without them).
    Kc = min(K, CALL_STEPS)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
           for _ in range(Kc)]
    for k in range(Kc):
        step(bufs0, evs[k])
    torch.cuda.synchronize(device)
    per_call = {}
    for j, nm in enumerate(names):
        ts = [evs[k][j].elapsed_time(evs[k][j + 1]) for k in range(Kc)]
        per_call[nm] = float(np.mean(ts))

    # e2e: the same step with its inputs in pinned host memory. Every step
    # uploads its CSR arrays, x and y0 and reads its five results back; the
    # uploads of step k+1 and the read-back of step k run on their own streams
    # while step k computes (two device buffer sets), as a pipelined user
    # would run it. Timed on the device from before the first upload to after
    # the last read-back.
    e2e = None
    if not args.no_e2e:
        hrp = torch.from_numpy(inp.row_ptrs).pin_memory()
        hci = torch.from_numpy(inp.col_idx).pin_memory()
        hva = torch.from_numpy(inp.value).pin_memory()
        hx = torch.from_numpy(inp.x).pin_memory()
        hy0 = torch.from_numpy(inp.y0).pin_memory()
        sets = [bufs0, make_bufs()]
        outs = [[torch.empty(R, dtype=torch.float32).pin_memory() for _ in FORMATS]
                for _ in sets]
        up_s, down_s = torch.cuda.Stream(device), torch.cuda.Stream(device)
        ready = [torch.cuda.Event() for _ in sets]
        done = [torch.cuda.Event() for _ in sets]
        freed = [torch.cuda.Event() for _ in sets]

        def upload(j):
            b = sets[j]
            with torch.cuda.stream(up_s):
                up_s.wait_event(freed[j])  # the set's previous results are read back
                b["rp"].copy_(hrp, non_blocking=True)
                b["ci"].copy_(hci, non_blocking=True)
                b["va"].copy_(hva, non_blocking=True)
                b["x"].copy_(hx, non_blocking=True)
                # y0 crosses once; the per-format accumulators are device copies
                b["ys"][FORMATS[0]].copy_(hy0, non_blocking=True)
                for f in FORMATS[1:]:
                    b["ys"][f].copy_(b["ys"][FORMATS[0]], non_blocking=True)
                ready[j].record(up_s)

        def download(j):
            with torch.cuda.stream(down_s):
                down_s.wait_event(done[j])
                for f, o in zip(FORMATS, outs[j]):
                    o.copy_(sets[j]["ys"][f], non_blocking=True)
                freed[j].record(down_s)

        def run(n, start_event=None):
            if start_event is not None:
                up_s.wait_event(start_event)
            upload(0)
            for k in range(n):
                if k + 1 < n:
                    upload((k + 1) % 2)
                stream.wait_event(ready[k % 2])
                step(sets[k % 2])
                done[k % 2].record(stream)
                download(k % 2)
            stream.wait_stream(down_s)

        run(max(3, args.warmup // 2))
        torch.cuda.synchronize(device)
        Ke = max(3, K // 4)
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run(Ke, e0)
        e1.record(stream)
        torch.cuda.synchronize(device)
        e_ms = allreduce_max(e0.elapsed_time(e1), world, device)
        h2d = 4 * (R + 1) + 8 * Z + 4 * C + 4 * R
        d2h = 4 * R * len(FORMATS)
        e2e = {"value": round(world * len(FORMATS) * compulsory_bytes(R, C, Z) * Ke
                              / (e_ms * 1e-3) / 1e9, 2),
               "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e_ms / Ke, 4), "steps": Ke,
               "pipelining": "uploads of step k+1 and read-back of step k overlap step k "
                             "(two device buffer sets, separate copy streams)"}

    if rank != 0:
        return None

    peak, peak_kind = load_peaks()
    step_ms = elapsed_ms / K
    spmv_bytes = len(FORMATS) * compulsory_bytes(R, C, Z)
    value = world * spmv_bytes / (step_ms * 1e-3) / 1e9
    gflops = world * len(FORMATS) * 2 * Z / (step_ms * 1e-3) / 1e9
    calls = {}
    for nm in names:
        b = call_bytes(nm, R, C, Z, info["ell_width"], info["hyb_width"], info["hyb_tail"])
        ms = per_call[nm]
        gbs = b / (ms * 1e-3) / 1e9 if ms > 0 else None
        calls[nm] = {"ms": round(ms, 5), "alg_bytes": b, "GB/s": round(gbs, 1),
                     "frac": round(gbs / peak, 4), "share": round(ms / step_ms, 4)}
        if nm.startswith("spmv_"):
            calls[nm]["GFLOP/s"] = round(2 * Z / (ms * 1e-3) / 1e9, 1)
    top = max(calls, key=lambda n: calls[n]["ms"])
    best_spmv = min((n for n in calls if n.startswith("spmv_")), key=lambda n: calls[n]["ms"])
    # The dominant kernel: from the workload's ncu launch list where one is
    # committed, else the single-kernel call with the longest event time.
    if args.workload in DOMINANT:
        dom_call, dom_kernel = DOMINANT[args.workload]
        dom_source = "largest share of the ncu launch list of this workload's step"
    else:
        dom_call = max(SINGLE_KERNEL_CALLS, key=lambda n: calls[n]["ms"])
        dom_kernel = SINGLE_KERNEL_CALLS[dom_call]
        dom_source = "longest single-kernel call by CUDA events (no launch list committed)"
    dom_traffic = traffic_record(args.workload, dom_kernel)
    roof = {"bound": "hbm", "kernel": dom_kernel, "kernel_call": dom_call,
            "kernel_source": dom_source,
            "achieved": calls[dom_call]["GB/s"], "peak": peak, "peak_kind": peak_kind,
            "unit": "GB/s", "frac": calls[dom_call]["frac"],
            "alg_bytes_per_launch": calls[dom_call]["alg_bytes"],
            "launch_us": round(calls[dom_call]["ms"] * 1e3, 2), "traffic": dom_traffic,
            "largest_call": {"call": top, "GB/s": calls[top]["GB/s"], "frac": calls[top]["frac"],
                             "share": calls[top]["share"]},
            "best_spmv": {"call": best_spmv, "GB/s": calls[best_spmv]["GB/s"],
                          "frac": calls[best_spmv]["frac"],
                          "GFLOP/s": calls[best_spmv]["GFLOP/s"]}}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded generator, seed 0)",
        "config": {"workload": f"{args.workload}: {WORKLOAD_DESC[args.workload]}",
                   "num_rows": R, "num_cols": C, "nnz": Z,
                   "step": "create+validate+stats, convert COO/ELL/HYB/JDS, select, "
                           "SpMV in CSR/COO/ELL/HYB/JDS",
                   "auto_format": info["auto"], "hyb_width": info["hyb_width"],
                   "l2": "no flush: each step moves > 1 GB, far beyond the 129 MB L2",
                   "parallelism": f"replicas x{world}"},
        "gflops": round(gflops, 1),
        "calls": calls,
        "calls_protocol": f"a separate pass of {min(K, CALL_STEPS)} steps with a CUDA event "
                          "between every two calls; mean per call",
        "roofline": roof,
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": e2e,
    }
    return line


class L2Flush:
    """Leaves L2 cold and clean: writes a buffer of twice the L2 size, then
    reads another one, so that L2 holds clean lines of neither the matrix nor
    the vectors (after the write alone, up to the whole L2 is dirty and the
    timed kernel pays its write-back: 34-40 MB more DRAM writes, ELL on
    stencil27 143 -> 158 us)."""

    def __init__(self, torch, device):
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        self.dirty = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=device)
        self.clean = torch.ones(2 * l2 // 4 + 1024, dtype=torch.float32, device=device)

    def __call__(self, tag=0.0):
        self.dirty.fill_(float(tag))
        self.clean.sum()

    def describe(self):
        n = self.dirty.numel() * 4
        return f"write {n} B, then read another {n} B (clean L2), before every run"


def cold_spmv_times(torch, m, f, x, y, y0, stream, flush, reps, warmup, warm=False):
    """Median ms of `reps` runs of one format's SpMV after `warmup` untimed
    ones: y reset to y0 and L2 flushed before every run, outside the CUDA
    events on the launching stream. warm=True: the same without the flush."""
    times = []
    for rep in range(warmup + reps):
        y.copy_(y0)  # y = y0 before every run, outside the events
        if not warm:
            flush(rep)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        m.run(f, x, y, stream=stream)
        e1.record(stream)
        e1.synchronize()
        if rep >= warmup:
            times.append(e0.elapsed_time(e1))
    return float(np.median(times))


def run_kernels(args, device):
    """Per-format SpMV timing on one workload: each rep resets y to y0 and
    flushes L2 (L2Flush) outside the timed events, then times one spmv_run
    with CUDA events on the launching stream; median over reps. Warm-L2 times
    (the same runs back to back without the flush) are reported apart. Each
    format's conversion from CSR: after one untimed conversion, the median of
    --convert-reps conversions, each after an L2 flush, against the
    conversion's algorithmic bytes (convert_bytes)."""
    import torch
    import spmv_sparse_storage_gb300 as sp
    inp = synth.make_workload(args.workload, seed=0)
    R, C, Z = inp.num_rows, inp.num_cols, inp.nnz
    stream = torch.cuda.current_stream(device)
    vdt = np.float64 if args.dtype == "f64" else np.float32
    vb = np.dtype(vdt).itemsize
    rp = torch.from_numpy(inp.row_ptrs).to(device)
    ci = torch.from_numpy(inp.col_idx).to(device)
    va = torch.from_numpy(inp.value.astype(vdt)).to(device)
    x = torch.from_numpy(inp.x.astype(vdt)).to(device)
    y0 = torch.from_numpy(inp.y0.astype(vdt)).to(device)
    y = y0.clone()
    flush = L2Flush(torch, device)
    peak, peak_kind = load_peaks()
    out = {}
    with sp.SparseMatrix(R, C, rp, ci, va, stream) as m:
        fmts = [f for f in args.formats.split(",") if f]
        conv_us = {}
        for f in fmts:
            if f == "CSR":
                continue
            try:
                m.convert(f, stream=stream, chunk_cols=args.chunk_cols)  # warm (pool, launches)
                ts = []
                for _ in range(args.convert_reps):
                    flush()
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    m.convert(f, stream=stream, chunk_cols=args.chunk_cols)
                    e1.record(stream)
                    e1.synchronize()
                    ts.append(e0.elapsed_time(e1) * 1e3)
                conv_us[f] = round(statistics.median(ts), 2)
            except sp.SpmvError as e:
                out[f] = {"error": str(e)}
        torch.cuda.synchronize(device)
        for f in fmts:
            if f in out:
                continue
            ms = cold_spmv_times(torch, m, f, x, y, y0, stream, flush, args.reps, args.warmup)
            ms_warm = cold_spmv_times(torch, m, f, x, y, y0, stream, flush, args.reps,
                                      args.warmup, warm=True)
            gbs = compulsory_bytes(R, C, Z, vb) / (ms * 1e-3) / 1e9
            gflops = 2 * Z / (ms * 1e-3) / 1e9
            gbs_warm = compulsory_bytes(R, C, Z, vb) / (ms_warm * 1e-3) / 1e9
            out[f] = {"us": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
                      "frac": round(gbs / peak, 4), "GFLOP/s": round(gflops, 1),
                      "convert_us": conv_us.get(f), "warm_l2_us": round(ms_warm * 1e3, 2),
                      "warm_l2_frac": round(gbs_warm / peak, 4)}
            if vb == 8:  # fp64 multiply-adds against the nominal 1.25 TFLOP/s fp64 rate
                out[f]["fp64_frac_nominal"] = round(gflops / FP64_NOMINAL_GFLOPS, 4)
            if f in ("ELL", "HYB", "SELL", "XBLOCK"):
                out[f]["slots"] = sp.spmv_export(m.handle, f)["ell_slots"]
            if f in conv_us:
                ex = sp.spmv_export(m.handle, f)
                cb = convert_bytes(f, R, C, Z, vb, width=ex.get("width", 0),
                                   tail=ex.get("coo_nnz", 0), slots=ex.get("ell_slots", 0))
                cgbs = cb / (conv_us[f] * 1e-6) / 1e9
                out[f].update({"convert_alg_bytes": cb, "convert_GB/s": round(cgbs, 1),
                               "convert_frac": round(cgbs / peak, 4)})
        sel = m.select()
    line = {"mode": "kernels", "workload": args.workload, "dtype": args.dtype, "rows": R,
            "nnz": Z,
            "l2_flush": flush.describe() + ", outside the events; warm_l2_*: the "
                        "same runs back to back without the flush",
            "reps": args.reps, "peak": peak,
            "peak_kind": peak_kind, "auto": sel, "kernels": out}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle_spmv(inp, inp.value.astype(vdt), inp.x.astype(vdt),
                                                inp.y0.astype(vdt))
    return line


def per_config_table(args, device, inputs):
    """Every format's SpMV alone on each of the five workloads, cold L2
    (cold_spmv_times: y reset, L2 flushed before every run), with the
    selector's choice and the fastest format. `inputs` maps workload names to
    already generated inputs (others are generated here)."""
    import torch
    import spmv_sparse_storage_gb300 as sp
    stream = torch.cuda.current_stream(device)
    flush = L2Flush(torch, device)
    peak, _ = load_peaks()
    table = {}
    for w in CONFIG_ORDER:
        inp = inputs.get(w) or synth.make_workload(w, seed=0)
        R, C, Z = inp.num_rows, inp.num_cols, inp.nnz
        cb = compulsory_bytes(R, C, Z)
        rp = torch.from_numpy(inp.row_ptrs).to(device)
        ci = torch.from_numpy(inp.col_idx).to(device)
        va = torch.from_numpy(inp.value).to(device)
        x = torch.from_numpy(inp.x).to(device)
        y0 = torch.from_numpy(inp.y0).to(device)
        y = y0.clone()
        fm = {}
        with sp.SparseMatrix(R, C, rp, ci, va, stream) as m:
            for f in ALL_FORMATS:
                try:
                    if f != "CSR":
                        m.convert(f, stream=stream)
                except sp.SpmvError as e:
                    fm[f] = {"error": str(e)}
                    continue
                ms = cold_spmv_times(torch, m, f, x, y, y0, stream, flush, args.config_reps,
                                     args.config_warmup)
                gbs = cb / (ms * 1e-3) / 1e9
                fm[f] = {"us": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
                         "frac": round(gbs / peak, 4),
                         "GFLOP/s": round(2 * Z / (ms * 1e-3) / 1e9, 1)}
            auto, width = m.select()
        timed = {f: v["us"] for f, v in fm.items() if "us" in v}
        best = min(timed, key=timed.get)
        table[w] = {"rows": R, "cols": C, "nnz": Z, "compulsory_bytes": cb, "formats": fm,
                    "auto": auto, "auto_hyb_width": width, "auto_us": timed.get(auto),
                    "best": best, "best_us": timed[best], "best_frac": fm[best]["frac"],
                    "auto_over_best": round(timed[auto] / timed[best], 4)
                    if auto in timed else None}
        del rp, ci, va, x, y0, y
        torch.cuda.empty_cache()
    return {"protocol": f"each format's spmv_run alone, median of {args.config_reps} runs after "
                        f"{args.config_warmup}; y reset and L2 flushed ({flush.describe()}) "
                        "before every run, outside the CUDA events; fraction of the measured "
                        "copy peak",
            "configs": table}


def cg_alg_bytes(R, slots):
    """Algorithmic HBM bytes of one CG iteration on the ELL path: the fused
    direction + SpMV kernel reads the slots (8 B each), g and d_old (4 B per
    row each, once) and writes d_new and q (4 B each); the update reads X, g,
    d_new, q and writes X, g (24 B per row)."""
    return 8 * slots + (16 + 24) * R


def run_cg(args, device):
    """Conjugate gradient for A·X + Y = 0 on the workload (ELL, tol 0 so that
    exactly --cg-iters iterations run): iterations per second from CUDA events
    around spmv_cg_solve on the launching stream (its periodic stop checks
    included), over --steps solves after --warmup."""
    import torch
    import spmv_sparse_storage_gb300 as sp
    inp = synth.make_workload(args.workload, seed=0)
    R, C, Z = inp.num_rows, inp.num_cols, inp.nnz
    stream = torch.cuda.current_stream(device)
    rp = torch.from_numpy(inp.row_ptrs).to(device)
    ci = torch.from_numpy(inp.col_idx).to(device)
    va = torch.from_numpy(inp.value).to(device)
    Y = torch.from_numpy(inp.y0).to(device)
    X = torch.zeros(R, dtype=torch.float32, device=device)
    iters = args.cg_iters
    peak, peak_kind = load_peaks()
    with sp.SparseMatrix(R, C, rp, ci, va, stream) as m:
        m.convert("ELL", stream=stream)
        slots = sp.spmv_export(m.handle, "ELL")["ell_slots"]
        for _ in range(args.warmup):
            X.zero_()
            m.cg_solve("ELL", Y, X, max_iter=iters, tol=0.0, stream=stream)
        torch.cuda.synchronize(device)
        clocks = ClockSampler(device.index if device.index is not None else 0)
        clocks.start()
        time.sleep(0.3)
        times = []
        launches0 = sp.spmv_launch_count()
        for _ in range(args.steps):
            X.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            info = m.cg_solve("ELL", Y, X, max_iter=iters, tol=0.0, stream=stream)
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        launches = (sp.spmv_launch_count() - launches0) // max(1, args.steps)
        clk = clocks.stop()
    ms = float(np.median(times))
    it_s = iters / (ms * 1e-3)
    b = cg_alg_bytes(R, slots)
    gbs = b * iters / (ms * 1e-3) / 1e9
    # CPU oracle: the same solve, a bounded number of iterations on the full matrix
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        orc = oracle.get()
        n_cpu = 5
        t = time.perf_counter()
        orc.cg(inp.row_ptrs, inp.col_idx, inp.value, inp.y0, None, max_iter=n_cpu, tol=0.0)
        dt = time.perf_counter() - t
        cpu = {"value": round(n_cpu / dt, 3), "unit": "iterations/s", "cores": 1,
               "kind": "oracle", "sample": f"{n_cpu} CG iterations on the full {args.workload} "
                                           "matrix (fp64, 1 thread), one run"}
    return {"mode": "cg", "metric": "CG iterations/s (A·X + Y = 0, fp32 vectors, ELL)",
            "value": round(it_s, 1), "unit": "iterations/s", "higher_is_better": True,
            "workload": f"{args.workload}: {WORKLOAD_DESC[args.workload]}",
            "iterations_per_solve": iters, "solves": args.steps, "ms_per_solve": round(ms, 4),
            "us_per_iteration": round(ms * 1e3 / iters, 2), "residual_ratio":
                round(info["residual_norm"] / max(info["y_norm"], 1e-300), 6),
            "gpu_launches_per_solve": launches,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": round(gbs / peak, 4),
                         "alg_bytes_per_iteration": b, "traffic": None},
            "cpu_baseline": cpu, "clocks": clk}


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(v, world, device):
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline object and the reference arm)
# ---------------------------------------------------------------------------
def oracle_step(orc, inp):
    """The whole path on the CPU oracle: validate, statistics, conversions,
    selection and the SpMV of every format (fp64 sums)."""
    rp, ci, va, x, y0 = inp.row_ptrs, inp.col_idx, inp.value, inp.x, inp.y0
    R = inp.num_rows
    orc.validate(R, inp.num_cols, rp, ci)
    st = orc.row_stats(rp)
    coo = orc.csr_to_coo(rp, ci, va)
    ell = orc.csr_to_ell(rp, ci, va)
    K = orc.hyb_auto_width(rp)
    hyb = orc.csr_to_hyb(rp, ci, va, K)
    jds = orc.csr_to_jds(rp, ci, va)
    orc.select(R, inp.num_cols, inp.nnz, st["max_len"], 0.0)
    orc.spmv_csr(rp, ci, va, x, y0)
    orc.spmv_coo(R, coo["row_idx"], coo["col_idx"], coo["value"], x, y0)
    orc.spmv_ell(ell, x, y0)
    orc.spmv_hyb(hyb, x, y0)
    orc.spmv_jds(jds, x, y0)


def row_sample(inp, rows):
    """The first `rows` rows of the workload (all their entries); x unchanged."""
    rows = min(rows, inp.num_rows)
    end = int(inp.row_ptrs[rows])
    return synth.CSRInput(inp.name + f"[:{rows}]", rows, inp.num_cols,
                          inp.row_ptrs[:rows + 1].copy(), inp.col_idx[:end].copy(),
                          inp.value[:end].copy(), inp.x, inp.y0[:rows].copy())


def host_cpu():
    """The host's core count and CPU model (lscpu's "Model name", else the
    platform's processor string), for labelling single-core oracle timings."""
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        import platform
        model = platform.processor() or platform.machine()
    return {"host_cores": os.cpu_count(), "cpu_model": model}


def time_oracle_spmv(inp, value, x, y0, reps=3):
    """The fp64 CSR SpMV oracle (plain C, one thread) on the whole matrix:
    median of `reps` runs, as effective GB/s of the same compulsory bytes."""
    import oracle
    orc = oracle.get()
    f64 = value.dtype == np.float64
    times = []
    for _ in range(reps):
        t = time.perf_counter()
        if f64:
            orc.spmv_csr_f64(inp.row_ptrs, inp.col_idx, value, x, y0)
        else:
            orc.spmv_csr(inp.row_ptrs, inp.col_idx, value, x, y0)
        times.append(time.perf_counter() - t)
    s_med = float(np.median(times))
    vb = 8 if f64 else 4
    gbs = compulsory_bytes(inp.num_rows, inp.num_cols, inp.nnz, vb) / s_med / 1e9
    host = host_cpu()
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"the whole matrix, CSR SpMV only, median of {reps} runs "
                      f"(1 core of {host['host_cores']})",
            "us": round(s_med * 1e6, 1), "GFLOP/s": round(2 * inp.nnz / s_med / 1e9, 4), **host}


def sample_bytes(sample):
    """Compulsory SpMV bytes of a row sample: value and column per nonzero,
    rowPtrs and y per row, and the x entries it reads once (the distinct
    columns its nonzeros reference; a row sample of a banded matrix reads only
    part of x)."""
    cols = int(np.unique(sample.col_idx).size) if sample.nnz else 0
    return 8 * sample.nnz + 12 * sample.num_rows + 4 * cols


def time_oracle(inp, budget_s, steps=None, warmup=0):
    """The oracle doing the step on a row sample of `inp`, sized so that the
    whole run takes about budget_s. With `steps`, `warmup` untimed steps and
    then exactly `steps` timed ones; without, timed steps until budget_s has
    passed (at least one)."""
    import oracle
    orc = oracle.get()
    # calibrate: the time per row of one step on a small sample
    probe = row_sample(inp, max(1, inp.num_rows // 64))
    t = time.perf_counter()
    oracle_step(orc, probe)
    per_row = (time.perf_counter() - t) / probe.num_rows
    n_steps = (steps + warmup) if steps else 5
    rows = int(min(inp.num_rows, max(1, (budget_s / n_steps) / max(per_row, 1e-12))))
    sample = row_sample(inp, rows)
    times = []
    if steps:
        for _ in range(warmup):
            oracle_step(orc, sample)
        for _ in range(steps):
            t = time.perf_counter()
            oracle_step(orc, sample)
            times.append(time.perf_counter() - t)
    else:
        t_end = time.perf_counter() + budget_s
        while not times or time.perf_counter() < t_end:
            t = time.perf_counter()
            oracle_step(orc, sample)
            times.append(time.perf_counter() - t)
    step_s = float(np.median(times))
    b = len(FORMATS) * sample_bytes(sample)
    return {"value": round(b / step_s / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"rows [0, {sample.num_rows}) of {inp.name} ({sample.nnz} nnz), "
                      f"whole path per step, median of {len(times)} timed steps"
                      + (f" after {warmup} untimed" if steps and warmup else "")
                      + "; bytes: 8 per nonzero, 12 per row, 4 per distinct column "
                        "the sample references (its share of x)",
            "ms_per_step": round(step_s * 1e3, 3), "steps": len(times), **host_cpu()}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    inp = synth.make_workload(args.workload, seed=0)
    budget = max(5.0, min(120.0, 0.5 * (args.steps + args.warmup)))
    cb = time_oracle(inp, budget_s=budget, steps=args.steps, warmup=args.warmup)
    line = {
        "impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "GB/s",
        "n_gpus": world, "steps": cb["steps"], "warmup": args.warmup,
        "ms_per_step": cb["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generator, seed 0)",
        "config": {"workload": f"{args.workload}: {WORKLOAD_DESC[args.workload]}",
                   "step": "the same path on the CPU oracle (plain C, fp64, 1 thread)",
                   "parallelism": "1 CPU core"},
        "cpu_baseline": {"value": cb["value"], "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": cb["sample"]},
        "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--mode", choices=["step", "kernels", "cg"], default="step",
                    help="step: the whole path (default); kernels: per-format SpMV, cold L2; "
                         "cg: conjugate-gradient iterations/s")
    ap.add_argument("--cg-iters", type=int, default=200)
    ap.add_argument("--dtype", choices=["f32", "f64"], default="f32",
                    help="--mode kernels: value and vector type")
    ap.add_argument("--chunk-cols", type=int, default=0,
                    help="XBLOCK chunk width B (0: the library default)")
    ap.add_argument("--formats", default="CSR,COO,ELL,HYB,JDS,SELL,XBLOCK")
    ap.add_argument("--reps", type=int, default=50)
    ap.add_argument("--convert-reps", type=int, default=5,
                    help="--mode kernels: conversions timed per format (median; L2 flushed "
                         "before each)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="step mode: skip the per-format table of the five workloads")
    ap.add_argument("--config-reps", type=int, default=10)
    ap.add_argument("--config-warmup", type=int, default=3)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    if rank == 0:
        import importlib.util
        path = os.path.join(ROOT, "spmv_sparse_storage_gb300", "_build.py")
        spec = importlib.util.spec_from_file_location("_spmv_build", path)
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()
    barrier(world)
    if args.mode in ("kernels", "cg"):
        if rank == 0:
            fn = run_kernels if args.mode == "kernels" else run_cg
            print(json.dumps(fn(args, device)), flush=True)
        return
    inp = synth.make_workload(args.workload, seed=0)
    line = run_ours(args, rank, world, device, inp)
    if rank == 0:
        if not args.no_per_config:
            line["per_config"] = per_config_table(args, device, {args.workload: inp})
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = time_oracle(inp, budget_s=args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
