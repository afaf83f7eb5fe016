#!/usr/bin/env python
"""Benchmark of the fused SwiGLU + MXFP8 cast on GB300.

One step = the six fused cells of the pages' headline shape M=131072,
N=8192 ("Add swiglu + MXFP8 fused CuTe DSL kernel", section "Performance"):
forward rowwise / colwise / both and backward rowwise / colwise / both, each
one launch of libmxfp8 over the same resident bf16 inputs (gate, up, dh:
3 x 2 GiB, far larger than L2, so no L2 flush is needed between steps).

The metric is algorithmic GB/s = (bytes read + bytes written) / time with
GB = 1e9: fwd reads 4MN and writes k(MN + MN/32), bwd reads 6MN and writes
2k(MN + MN/32), k = 1 (row or col) or 2 (both).  ``value`` is the whole
step's bytes over its time, summed over ranks (weak scaling: every rank casts
its own batch; no collective on the data path).

Prints one JSON line.  ``--impl reference`` instead times the CPU oracle on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

M_LARGE, N_LARGE = 131072, 8192
CELLS = [("fwd", 1), ("fwd", 2), ("fwd", 3), ("bwd", 1), ("bwd", 2), ("bwd", 3)]
MODE_NAME = {1: "row", 2: "col", 3: "both"}
METRIC = "fused SwiGLU+MXFP8 cast GB/s (fwd/bwd, row/col/both) and % of GB300 HBM peak"
WORKLOAD = "swiglu_mxfp8_fwd_bwd_row_col_both_131072x8192"
# the pages' own figures for these six cells at (131072, 8192), GB200 with
# clocks pinned at 2062 MHz (context, another machine): microseconds per cell
PAGES_US = {("fwd", 1): 904.19, ("fwd", 2): 1022.98, ("fwd", 3): 1216.08,
            ("bwd", 1): 1321.98, ("bwd", 2): 1710.08, ("bwd", 3): 1859.09}


# DRAM traffic (read + write bytes) of one full-size launch of each kernel,
# measured by ncu on that launch alone (dram__bytes_read.sum +
# dram__bytes_write.sum, a one-pass capture, in a separate run of this
# script's --cell mode: a number taken under a profiler is not timed here);
# keyed to the hash of the kernel sources it was taken on (None once they
# change).
TRAFFIC = {
    "bwd_both": (10.8328e9, "4a518d3dad333b0d"),
    "bwd_both_gelu": (10.845e9, "4a518d3dad333b0d"),
    "bwd_col": (8.63175e9, "4a518d3dad333b0d"),
    "bwd_row": (8.63187e9, "4a518d3dad333b0d"),
    "fwd_both": (6.47681e9, "4a518d3dad333b0d"),
    "fwd_col": (5.38253e9, "4a518d3dad333b0d"),
    "fwd_row": (5.38212e9, "4a518d3dad333b0d"),
    "fwd_row_gelu": (5.38247e9, "4a518d3dad333b0d"),
    "quant3d": (8.105e9, "4a518d3dad333b0d"),
    "quant_both": (4.31589e9, "4a518d3dad333b0d"),
    "quant_row": (3.22182e9, "4a518d3dad333b0d"),
}
TRAFFIC_KIND = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one full-size launch of the kernel, "
                "captured alone in a separate run (bench.py --cell <cell> --steps 1 --warmup 0)")


def kernel_source_hash() -> str:
    import glob
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mxfp8_quantization_moe_gb300", "csrc")
    files = [os.path.join(csrc, n) for n in ("device.cuh", "kernel.cuh", "launch.cuh")]
    files += sorted(glob.glob(os.path.join(csrc, "ops_*.cu")))
    for f in files:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(cell: str):
    t = TRAFFIC.get(cell)
    if t is None or t[1] != kernel_source_hash():
        return None
    return t[0]


def configs_note(steps: int) -> str:
    """How the per-workload lines of the bench line were measured."""
    return ("each workload of the pages' shape list, one cell at a time: median of %d "
            "CUDA-event launch times, inputs resident, L2 flushed before each launch "
            "(a 512 MB write, then a 1 GB read so the written lines leave L2 outside "
            "the timed launch); 3D = the first E experts of the seed-4 draw; "
            "the mixed workload scales every 7th row by up to 2^20, so about 5 %% of "
            "its 8-element chunks hold a gate below the fast range, settled pair by "
            "pair on the exact path; the (128, 128) forward is launch-bound" % steps)


def cell_bytes(kind: str, mode: int, M: int, N: int) -> int:
    k = 2 if mode == 3 else 1
    mn = M * N
    cast = mn + mn // 32
    return 4 * mn + k * cast if kind == "fwd" else 6 * mn + 2 * k * cast


def step_bytes(M=M_LARGE, N=N_LARGE) -> int:
    return sum(cell_bytes(k, m, M, N) for k, m in CELLS)


def pages_step_gbs() -> float:
    return step_bytes() / (sum(PAGES_US.values()) * 1e-6) / 1e9


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def base_config(extra=None):
    c = {"workload": WORKLOAD, "M": M_LARGE, "N": N_LARGE,
         "cells": ["%s_%s" % (k, MODE_NAME[m]) for k, m in CELLS],
         "inputs": "gate, up, dh bf16 N(0,1), seed 3 (+rank), resident in HBM",
         "l2": "no flush: 6 GiB of inputs per step, far above the 129 MB L2"}
    if extra:
        c.update(extra)
    return c


# ------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        with open(self.f.name) as fh:
            lines = [ln.strip() for ln in fh if ln.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- CPU oracle
def oracle_step(gate_b, up_b, dh_b, threads=None):
    """The six cells of one step through the CPU oracle (plain definitions)."""
    import oracle as O
    for kind, mode in CELLS:
        if kind == "fwd":
            O.swiglu_fwd(gate_b, up_b, mode, threads=threads)
        else:
            O.swiglu_bwd(dh_b, gate_b, up_b, mode, threads=threads)


def cpu_sample(rows: int, seed: int = 3):
    """A (rows, 8192) sample of the workload drawn on the host (same recipe)."""
    import numpy as np
    import torch
    import synthetic
    g = torch.Generator().manual_seed(seed)
    t = [synthetic.normal_bf16((rows, N_LARGE), 1.0, g, "cpu") for _ in range(3)]
    return [x.view(torch.int16).numpy().view(np.uint16) for x in t]


def time_oracle(target_s: float, threads: int):
    """Grow a sample of 32-row blocks until one oracle step takes ~target_s."""
    rows = 32
    while True:
        gate, up, dh = cpu_sample(rows)
        t0 = time.perf_counter()
        oracle_step(gate, up, dh, threads=threads)
        dt = time.perf_counter() - t0
        if dt >= target_s * 0.5 or rows >= 4096:
            return rows, dt
        rows = min(4096, max(rows * 2, int(rows * target_s / max(dt, 1e-3)) // 32 * 32))


def cpu_baseline(target_s: float):
    """The oracle on all host cores, then on one thread (a smaller sample)."""
    threads = os.cpu_count() or 1
    rows, dt = time_oracle(target_s, threads)
    b = step_bytes(rows, N_LARGE)
    rows1, dt1 = time_oracle(target_s / 2, 1)
    b1 = step_bytes(rows1, N_LARGE)
    return {"value": b / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "%d of 131072 rows (%d 32-row blocks) x 8192, all six cells, one pass, "
                      "%.1f s on %d threads" % (rows, rows // 32, dt, threads),
            "single_thread": {"value": b1 / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": "%d of 131072 rows x 8192, all six cells, one pass, %.1f s"
                                        % (rows1, dt1)}}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    threads = os.cpu_count() or 1
    if args.ref_blocks > 0:
        rows = 32 * args.ref_blocks
    else:
        # a sample per step sized so that all the steps take about
        # --ref-seconds (tiny samples measure the thread pool, not the oracle)
        rows, _ = time_oracle(args.ref_seconds / max(1, args.steps + args.warmup), threads)
    gate, up, dh = cpu_sample(rows)
    for _ in range(args.warmup):
        oracle_step(gate, up, dh, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(gate, up, dh, threads=threads)
    dt = time.perf_counter() - t0
    b = step_bytes(rows, N_LARGE)
    val = b * args.steps / dt / 1e9
    sample = "%d of 131072 rows x 8192 per step, all six cells, %d threads" % (rows, threads)
    line = {"metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": base_config({"sample_rows": rows}), "impl": "reference",
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------------- GPU
def slowest_rank_seconds(elapsed: float, world: int, device) -> float:
    """The job's time for a timed region: the slowest rank's (MAX over the
    default process group; one rank: its own)."""
    if world <= 1:
        return elapsed
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job rate: every rank processed its own units (weak scaling), so
    the bytes of all ranks over the slowest rank's time."""
    return bytes_per_rank * world / seconds / 1e9


# ------------------------------------------------------ every config's cells
L2_FLUSH_BYTES = 512 * 2 ** 20       # > 2 x the 129 MB L2


def time_launches(fn, steps: int, warmup: int, flush=None) -> float:
    """Median CUDA-event time (us) of one launch of ``fn`` over ``steps``
    launches after ``warmup`` untimed ones; ``flush`` runs before each timed
    launch, outside its events."""
    import torch
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        if flush is not None:
            flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) * 1e3 for a, b in evs)


def quant3d_bytes(E: int, N: int, K: int) -> int:
    return E * N * K * 2 + E * N * K + E * N * K // 32


def measure_configs(mx, synthetic, peak: float, steps: int, warmup: int):
    """Every workload of the pages' shape list, one cell at a time: the median
    launch time over ``steps`` launches, inputs resident in HBM, L2 flushed
    before each launch.  Keys: workload/cell."""
    import torch
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    clean_buf = torch.zeros(L2_FLUSH_BYTES // 2, dtype=torch.int32, device="cuda")
    clean_out = torch.empty((), dtype=torch.int64, device="cuda")

    def flush():
        # write a buffer larger than L2, then read another one, so that the
        # written lines are written back here and not inside the timed launch
        flush_buf.zero_()
        torch.sum(clean_buf, dim=0, dtype=torch.int64, out=clean_out)

    rows = {}

    def record(key, fn, nbytes):
        us = time_launches(fn, steps, warmup, flush)
        rows[key] = {"us": round(us, 2), "GBps": round(nbytes / us / 1e3, 1),
                     "frac_of_peak": round(nbytes / us / 1e3 / peak, 4), "bytes": nbytes}

    def fused_cells(name, gate, up, dh, cells):
        M, N = gate.shape
        for kind, mode in cells:
            if kind == "fwd":
                o = mx._alloc(M, N, mode, gate.device)
                fn = lambda o=o, mode=mode: mx.swiglu_fwd(gate, up, mode, out=o)
            else:
                o = mx.swiglu_bwd(dh, gate, up, mode)
                fn = lambda o=o, mode=mode: mx.swiglu_bwd(dh, gate, up, mode, out=o)
            record("%s/%s_%s" % (name, kind, MODE_NAME[mode]), fn, cell_bytes(kind, mode, M, N))
            del o

    buf, gate, up = synthetic.fwd_128x128(device="cuda")
    fused_cells("fwd_128x128", gate, up, None, [("fwd", 1)])
    g, u, d = synthetic.mixed(device="cuda")
    fused_cells("mixed_4096x7168", g, u, d, [("fwd", 3), ("bwd", 3)])
    del g, u, d
    g, u, d = synthetic.outlier(device="cuda")
    fused_cells("outlier_16384x7168", g, u, d, CELLS)
    del g, u, d
    x = synthetic.experts(64, device="cuda")
    _, N, K = x.shape
    for E in (1, 4, 16, 64):
        xe = x[:E]
        q = torch.empty((E, K, N), dtype=torch.uint8, device="cuda")
        sc = torch.empty((E, N // 32, K), dtype=torch.uint8, device="cuda")
        record("experts_E%d/quant3d_col" % E, lambda xe=xe, q=q, sc=sc: mx.quant_3d_colwise(xe, q, sc),
               quant3d_bytes(E, N, K))
        del q, sc
    del x, flush_buf, clean_buf
    torch.cuda.empty_cache()
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mx", choices=["mx", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-slabs", type=int, default=8,
                    help="row slabs the end-to-end step is pipelined over")
    ap.add_argument("--e2e-copy-streams", type=int, default=1,
                    help="streams per copy direction in the end-to-end step")
    ap.add_argument("--ref-blocks", type=int, default=0,
                    help="reference arm: 32-row blocks per step (0: sized by --ref-seconds)")
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="reference arm: about how long all its steps take")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config cell timings (every workload of the pages' shape list)")
    ap.add_argument("--config-steps", type=int, default=20)
    ap.add_argument("--cell", default=None,
                    help="time one cell only (fwd_row ... bwd_both, quant_row/col/both, quant3d, "
                         "quant3d_row/both) "
                         "on --rows rows; prints per-launch microseconds (for profiling)")
    ap.add_argument("--rows", type=int, default=M_LARGE)
    ap.add_argument("--experts", type=int, default=64)
    ap.add_argument("--blocked", action="store_true",
                    help="with --cell: scales in the blocked 128 x 4 tile layout")
    ap.add_argument("--keep-h", action="store_true",
                    help="with --cell fwd_row / fwd_both: also write the bf16 activation")
    ap.add_argument("--groups", type=int, default=0,
                    help="with --cell quant_* / fwd_* / bwd_*: per-group blocked scales for this many "
                         "token groups of random 32-row-aligned sizes")
    ap.add_argument("--act", default="silu", choices=["silu", "gelu"],
                    help="with --cell fwd_* / bwd_*: the gated activation (gelu: GEGLU)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.cell:
        return run_cell(args)

    import torch
    import torch.distributed as dist

    # the CPU oracle's thread pool is started before any GPU work
    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(args.cpu_seconds)

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import mxfp8_quantization_moe_gb300 as mx
    import synthetic

    mx.init()
    gate, up, dh = synthetic.large(device="cuda", seed=synthetic.SEEDS["large_131072x8192"] + rank)
    M, N = gate.shape
    fwd_out = {m: mx._alloc(M, N, m, gate.device) for m in (1, 2, 3)}
    bwd_out = {}
    for m in (1, 2, 3):
        o = mx.SwiGLUGrads()
        if m & 1:
            o.q_row = torch.empty((M, 2 * N), dtype=torch.uint8, device="cuda")
            o.s_row = torch.empty((M, 2 * N // 32), dtype=torch.uint8, device="cuda")
        if m & 2:
            o.q_col = torch.empty((2 * N, M), dtype=torch.uint8, device="cuda")
            o.s_col = torch.empty((M // 32, 2 * N), dtype=torch.uint8, device="cuda")
        bwd_out[m] = o
    stream = torch.cuda.current_stream()

    def launch(kind, mode):
        if kind == "fwd":
            mx.swiglu_fwd(gate, up, mode, out=fwd_out[mode])
        else:
            mx.swiglu_bwd(dh, gate, up, mode, out=bwd_out[mode])

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        for c in CELLS:
            launch(*c)
    barrier()
    mx.device_status(reset=True)

    K = args.steps
    ev = {c: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)] for c in CELLS}
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    time.sleep(0.3)
    barrier()
    t_start.record(stream)
    for k in range(K):
        for c in CELLS:
            ev[c][k][0].record(stream)
            launch(*c)
            ev[c][k][1].record(stream)
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    elapsed = slowest_rank_seconds(t_start.elapsed_time(t_end) / 1e3, world, "cuda")
    flags, fallbacks = mx.device_status()
    if flags:
        raise SystemExit("device status flags %#x after the timed region" % flags)

    peak, peak_kind = peaks()
    per_cell = {}
    for c in CELLS:
        us = statistics.mean(a.elapsed_time(b) for a, b in ev[c]) * 1e3
        b = cell_bytes(c[0], c[1], M, N)
        per_cell["%s_%s" % (c[0], MODE_NAME[c[1]])] = {
            "us": round(us, 2), "GBps": round(b / us / 1e3, 1), "frac_of_peak": round(b / us / 1e3 / peak, 4),
            "bytes": b}
    dom = max(per_cell, key=lambda k: per_cell[k]["us"])
    dom_achieved = per_cell[dom]["GBps"]

    value = job_gbs(step_bytes(M, N) * K, world, elapsed)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, mx, gate, up, dh, fwd_out, bwd_out, launch, barrier, world)

    configs = None
    if not args.no_configs and rank == 0:
        del fwd_out, bwd_out
        torch.cuda.empty_cache()
        configs = measure_configs(mx, synthetic, peak, args.config_steps, max(3, args.warmup))
        flags, _ = mx.device_status()
        if flags:
            raise SystemExit("device status flags %#x after the per-config timings" % flags)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(elapsed / K * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": round(value / world / pages_step_gbs(), 4),
        "dtype": "f32", "data": "synthetic",
        "config": base_config({"parallelism": "replicas%d" % world if world > 1 else "single",
                               "vs_baseline_note": "pages' six-cell aggregate %.1f GB/s on GB200 "
                                                   "(another machine; context)" % pages_step_gbs()}),
        "frac_of_peak": round(value / world / peak, 4),
        "per_cell": per_cell,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": dom_achieved, "peak": peak,
                     "peak_kind": "%s hbm_gbs (copy)" % peak_kind, "unit": "GB/s",
                     "frac": round(dom_achieved / peak, 4), "traffic": traffic_for(dom),
                     "traffic_kind": TRAFFIC_KIND, "algorithmic_bytes": per_cell[dom]["bytes"]},
        "gpu_launches": K * len(CELLS),
        "fallback_elements": fallbacks,
        "clocks": clk,
    }
    if e2e:
        line["e2e"] = e2e
    if configs:
        line["configs"] = configs
        line["configs_note"] = configs_note(args.config_steps)
    if cpu:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_cell(args):
    """Time one kernel alone (used for ncu captures and tuning sweeps)."""
    import torch
    import mxfp8_quantization_moe_gb300 as mx
    import synthetic
    mx.init()
    kind, _, mname = args.cell.partition("_")
    mode = {"row": 1, "col": 2, "both": 3}.get(mname, 2)
    if args.blocked:
        mode |= mx.MXFP8_BLOCKED_SCALES
    if kind == "quant3d" and mname in ("row", "both") or (kind == "quant3d" and args.blocked):
        # mxfp8_quant_3d: rowwise / colwise / both, plain or per-expert blocked scales
        x = synthetic.experts(args.experts, device="cuda")
        E, N, K = x.shape
        k = 2 if mode & 3 == 3 else 1
        nbytes = E * N * K * 2 + k * (E * N * K + E * N * K // 32)
        out = mx.quant_3d(x, mode)
        fn = lambda: mx.quant_3d(x, mode, out=out)
    elif kind == "quant3d":
        x = synthetic.experts(args.experts, device="cuda")
        E, N, K = x.shape
        q = torch.empty((E, K, N), dtype=torch.uint8, device="cuda")
        s = torch.empty((E, N // 32, K), dtype=torch.uint8, device="cuda")
        nbytes = E * N * K * 2 + E * N * K + E * N * K // 32
        fn = lambda: mx.quant_3d_colwise(x, q, s)
    else:
        gate, up, dh = synthetic.large(M=args.rows, N=N_LARGE, device="cuda")
        M, N = gate.shape
        ends = None
        if args.groups:
            gen = torch.Generator().manual_seed(11)
            cuts = torch.randperm(M // 32 - 1, generator=gen)[:args.groups - 1].add(1).sort().values * 32
            ends = torch.cat([cuts, torch.tensor([M])]).to(torch.int32).cuda()
        if kind == "quant" and ends is not None:
            k = 2 if mode & 3 == 3 else 1
            nbytes = 2 * M * N + k * (M * N + M * N // 32)
            out = mx.quant_2d_grouped(gate, ends, mode & 3)
            fn = lambda: mx.quant_2d_grouped(gate, ends, mode & 3, out=out)
        elif kind == "fwd" and ends is not None:
            nbytes = cell_bytes("fwd", mode & 3, M, N)
            out = mx.swiglu_fwd_grouped(gate, up, ends, mode & 3, act=args.act)
            fn = lambda: mx.swiglu_fwd_grouped(gate, up, ends, mode & 3, act=args.act, out=out)
        elif ends is not None:
            nbytes = cell_bytes("bwd", mode & 3, M, N)
            out = mx.swiglu_bwd_grouped(dh, gate, up, ends, mode & 3, act=args.act)
            fn = lambda: mx.swiglu_bwd_grouped(dh, gate, up, ends, mode & 3, act=args.act, out=out)
        elif kind == "quant":
            out = mx._alloc(M, N, mode, gate.device)
            k = 2 if mode & 3 == 3 else 1
            nbytes = 2 * M * N + k * (M * N + M * N // 32)
            fn = lambda: mx.quant_2d(gate, mode, out=out)
        elif kind == "fwd":
            out = mx._alloc(M, N, mode, gate.device)
            nbytes = cell_bytes("fwd", mode & 3, M, N) + (2 * M * N if args.keep_h else 0)
            fn = lambda: mx.swiglu_fwd(gate, up, mode, out=out, keep_h=args.keep_h, act=args.act)
        else:
            out = mx.swiglu_bwd(dh, gate, up, mode, act=args.act)
            nbytes = cell_bytes("bwd", mode & 3, M, N)
            fn = lambda: mx.swiglu_bwd(dh, gate, up, mode, out=out, act=args.act)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in evs:
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 for a, b in evs]
    flags, fb = mx.device_status()
    peak, _ = peaks()
    med = statistics.median(us)
    print(json.dumps({"cell": args.cell + ("+blocked" if args.blocked else "") + ("+h" if args.keep_h else "")
                      + ("+gelu" if args.act == "gelu" else "")
                      + ("+groups%d" % args.groups if args.groups else ""),
                      "rows": args.rows,
                      "us_median": round(med, 2),
                      "us_min": round(min(us), 2), "GBps": round(nbytes / med / 1e3, 1),
                      "frac_of_peak": round(nbytes / med / 1e3 / peak, 4), "bytes": nbytes,
                      "flags": flags, "fallbacks": fb}), flush=True)
    return 0 if flags == 0 else 1


def run_e2e(args, mx, gate, up, dh, fwd_out, bwd_out, launch, barrier, world):
    """Same metric through the public API with host buffers: every step copies
    the inputs host->device from pinned memory, runs the six cells, and
    copies every cast output back to pinned host memory.  The step is
    pipelined over row slabs on three streams (host->device copies, the
    casts, device->host copies; events order each slab's stages and keep a
    slab's buffers from being overwritten while the previous step still
    reads them), so the two copy directions and the casts overlap.  Each
    slab has its own outputs: rowwise data and both scale sets are the
    slab's rows of the whole-tensor layouts; colwise data are column-major
    per slab."""
    import torch
    M, N = gate.shape
    S = max(1, args.e2e_slabs)
    while M % (32 * S):
        S -= 1
    Ms = M // S
    dev = gate.device
    h_in = [t.cpu().pin_memory() for t in (gate, up, dh)]

    def alloc_slab():
        f, b = {}, {}
        for m in (1, 2, 3):
            o = mx.MXFP8Cast()
            if m & 1:
                o.q_row = torch.empty((Ms, N), dtype=torch.uint8, device=dev)
                o.s_row = torch.empty((Ms, N // 32), dtype=torch.uint8, device=dev)
            if m & 2:
                o.q_col = torch.empty((N, Ms), dtype=torch.uint8, device=dev)
                o.s_col = torch.empty((Ms // 32, N), dtype=torch.uint8, device=dev)
            f[m] = o
            g = mx.SwiGLUGrads()
            if m & 1:
                g.q_row = torch.empty((Ms, 2 * N), dtype=torch.uint8, device=dev)
                g.s_row = torch.empty((Ms, 2 * N // 32), dtype=torch.uint8, device=dev)
            if m & 2:
                g.q_col = torch.empty((2 * N, Ms), dtype=torch.uint8, device=dev)
                g.s_col = torch.empty((Ms // 32, 2 * N), dtype=torch.uint8, device=dev)
            b[m] = g
        return f, b

    slabs = [alloc_slab() for _ in range(S)]
    outs = []       # per slab: device output tensors
    for f, b in slabs:
        outs.append([t for m in (1, 2, 3) for o in (f[m], b[m])
                     for t in (o.q_row, o.s_row, o.q_col, o.s_col) if t is not None])
    h_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in o] for o in outs]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for o in h_out for t in o)
    C = max(1, args.e2e_copy_streams)
    s_ins = [torch.cuda.Stream() for _ in range(C)]
    s_outs = [torch.cuda.Stream() for _ in range(C)]
    s_run = torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(S)]
    ev_run = [torch.cuda.Event() for _ in range(S)]
    ev_out = [torch.cuda.Event() for _ in range(S)]
    started = [False] * S

    def step():
        for k in range(S):
            r0, r1 = k * Ms, (k + 1) * Ms
            d_in = [t[r0:r1] for t in (gate, up, dh)]
            s_in, s_out = s_ins[k % C], s_outs[k % C]
            with torch.cuda.stream(s_in):
                if started[k]:
                    s_in.wait_event(ev_run[k])        # the previous step's casts read these rows
                for d, h in zip(d_in, h_in):
                    d.copy_(h[r0:r1], non_blocking=True)
                ev_in[k].record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(ev_in[k])
                if started[k]:
                    s_run.wait_event(ev_out[k])       # the previous step's copies read the outputs
                f, b = slabs[k]
                for kind, mode in CELLS:
                    if kind == "fwd":
                        mx.swiglu_fwd(d_in[0], d_in[1], mode, out=f[mode], stream=s_run)
                    else:
                        mx.swiglu_bwd(d_in[2], d_in[0], d_in[1], mode, out=b[mode], stream=s_run)
                ev_run[k].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[k])
                for d, h in zip(outs[k], h_out[k]):
                    h.copy_(d, non_blocking=True)
                ev_out[k].record(s_out)
            started[k] = True

    main = torch.cuda.current_stream()

    def join():
        for st in s_ins + [s_run] + s_outs:
            main.wait_stream(st)

    step()
    join()
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(1, args.e2e_steps)
    a.record(main)
    for st in s_ins + [s_run] + s_outs:
        st.wait_stream(main)
    for _ in range(n):
        step()
    join()
    b.record(main)
    barrier()
    el = slowest_rank_seconds(a.elapsed_time(b) / 1e3, world, "cuda")
    val = job_gbs(step_bytes() * n, world, el)
    return {"value": round(val, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n, "ms_per_step": round(el / n * 1e3, 3), "slabs": S,
            "note": "pipelined over %d row slabs: %d host->device, 1 cast and %d device->host streams; "
                    "per-slab outputs: rowwise data and both scale sets are the slab's rows of the "
                    "whole-tensor layouts, colwise data is column-major per slab ((N, M/%d) each) rather "
                    "than the (N, M) layout of one call" % (S, C, C, S)}


if __name__ == "__main__":
    sys.exit(main())
