"""Benchmark of one GQA decode step (KV-cache HBM GB/s and decode steps/s).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                    [--secondary NAME|none] [--variant ...] [--repeat-seconds S]

One step = one gqa_decode call on the workload's whole batch (one layer), with
the bf16 KV cache resident in HBM: the decode kernel plus the split-combine
kernel that follows it (programmatic dependent launch).  GB/s counts
algorithmic bytes only: the attended K and V rows,
sum_b seq_lens[b] * G * d * 2 bytes * 2.  The headline workload is the
Llama-3-70B-shaped batch (the largest single-GPU configuration); the
Mistral-7B-shaped step is measured in the same run and reported beside it
("secondary").

L2: inputs larger than L2.  The K/V caches are held in C copies and step i
reads copy i % C, with C chosen so that the C - 1 steps between two reads of a
copy stream at least three L2 capacities of other data; no step finds its
cache in L2.  (A write-flush between steps is not used: the dirty lines it
leaves slow the next kernel down by write-back traffic that is not its own.)

Timing: after W warm-up steps, K steps are captured in a CUDA graph (calls
through the public API, captured on one stream; the copy schedule continues
across replays).  A block = one replay = K steps back to back between its own
pair of CUDA events; R blocks run back to back (R chosen so that they take
about --repeat-seconds, for the clock samples), and ms_per_step = the median
block / K.  The read-bandwidth ceiling (a read-only TMA stream with the decode's
boxes, libgqa_b300_bench.so) is measured in the same run.

``--variant meanpool`` times the K/V mean-pool conversion instead; ``--variant
readonly`` prints the read-only stream's own line.

Under torchrun (N > 1) every rank runs an independent replica of the step on
its own GPU (nothing is sharded); value = bytes of all ranks / max time.

``--impl reference`` times the float64 CPU oracle on the host cores instead, on
a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from kv_cache_decode_06_b300.inputs import (  # noqa: E402
    CONFIGS, MEANPOOL_T5XXL, MEANPOOL_T5XXL_CHECKPOINT, MEANPOOL_TINY, T5XXL_SWEEP_GS, make_decode_inputs, make_meanpool_input,
    make_new_rows, make_paged_layout,
)

METRIC = "GQA decode KV-cache HBM GB/s (% of B300 peak) and decode steps/s, 1 GPU"
MEANPOOL_METRIC = "GQA K/V mean-pool conversion HBM GB/s (% of B300 peak), 1 GPU"
UNIT = "GB/s"
L2_COPIES_SPAN = 3            # L2 capacities streamed between two reads of one cache copy
CPU_BASELINE_SECONDS = 10.0   # host time spent on the float64 oracle for the cpu_baseline field
FALLBACK_HBM_GBS = 6400.0


MEANPOOL_DEFAULT = "t5xxl_checkpoint"


def meanpool_workload(name: str):
    """Shape of one mean-pool conversion call: one projection of one layer ([H, h, d_model]),
    or a whole checkpoint's K and V projections in one strided call ([outer, H, h * d_model])."""
    if name == "tiny":
        return "meanpool_tiny", dict(MEANPOOL_TINY)
    if name == "t5xxl_checkpoint":
        return "meanpool_t5xxl_checkpoint", dict(MEANPOOL_T5XXL_CHECKPOINT)
    if name.startswith("t5xxl_sweep_G"):
        d = dict(MEANPOOL_T5XXL)
        d["G"] = int(name.split("_G")[1])
        return f"meanpool_t5xxl_G{d['G']}", d
    raise SystemExit(f"--variant meanpool takes --workload tiny, t5xxl_checkpoint or t5xxl_sweep_G<g>, not {name}")


def workload(name: str):
    if name.startswith("t5xxl_sweep_G"):
        return CONFIGS["t5xxl_sweep"].with_G(int(name.split("_G")[1]))
    return CONFIGS[name]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# Source files of a kernel that has a file of its own; every other kernel is
# hashed over all of csrc except those files.
KERNEL_SOURCES = {"meanpool_kernel": ("meanpool.cu", "launch.h")}


def kernel_source_hash(kernel: str = "gqa_decode_tc_kernel") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kv_cache_decode_06_b300", "csrc")
    own = {fn for srcs in KERNEL_SOURCES.values() for fn in srcs if fn.endswith(".cu")}
    for fn in sorted(os.listdir(csrc)):
        if not fn.endswith((".cu", ".cuh", ".h")):
            continue
        if kernel in KERNEL_SOURCES:
            if fn not in KERNEL_SOURCES[kernel]:
                continue
        elif fn in own:
            continue
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, wl: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}__{wl}.md")
    try:
        txt = open(path).read()
    except OSError:
        return None
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)\s+source_hash:\s*([0-9a-f]+)", txt)
    if not m or m.group(2) != kernel_source_hash(kernel):
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm, smax = [], []
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for nm, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_oracle_step(inp, segments, window=0):
    """Time the float64 oracle on the rows of the given (b, g) segments; returns (seconds, kv bytes)."""
    import oracle
    cfg = inp.cfg
    rows = np.array([b * cfg.H + g * cfg.n + h for (b, g) in segments for h in range(cfg.n)], dtype=np.int64)
    att = [min(int(inp.seq_lens[b]), window) if window else int(inp.seq_lens[b]) for (b, _) in segments]
    kv = sum(att) * cfg.d * 2 * 2
    t0 = time.perf_counter()
    oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, rows=rows, window=window)
    return time.perf_counter() - t0, kv


def all_segments(cfg):
    return [(b, g) for b in range(cfg.B) for g in range(cfg.G)]


def cpu_oracle_rows(inp, rows):
    """Time the float64 oracle on the given output rows (b*H + i); returns (seconds, kv bytes).

    A row's share of the algorithmic bytes is its sequence's K+V rows divided by the
    n = H/G query heads that share them.
    """
    import oracle
    cfg = inp.cfg
    kv = sum(int(inp.seq_lens[r // cfg.H]) for r in rows) * cfg.d * 2 * 2 / cfg.n
    t0 = time.perf_counter()
    oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, rows=np.asarray(rows, dtype=np.int64))
    return time.perf_counter() - t0, kv


def run_reference(args, rank: int) -> None:
    """The float64 CPU oracle as the reference arm, rank 0 only.

    Each step is a bounded sample of the workload's output rows (at least one), sized
    so that the whole --steps/--warmup run spends about 150 s in the oracle.
    """
    if rank != 0:
        return
    import oracle
    if args.variant == "meanpool":
        run_reference_meanpool(args)
        return
    cfg = workload(args.workload or "llama3_70b")
    inp = make_decode_inputs(cfg, poison_tail=False)
    nrows_all = cfg.B * cfg.H
    cores = oracle.num_threads()
    # calibrate: seconds per row on this host (a whole group of rows, to use the threads)
    t, _ = cpu_oracle_rows(inp, list(range(min(nrows_all, cfg.n))))
    per_row = max(t / min(nrows_all, cfg.n), 1e-5)
    budget = 150.0 / max(1, args.steps + args.warmup)
    nrow = int(max(1, min(nrows_all, budget / per_row)))
    order = np.random.default_rng(0).permutation(nrows_all)
    for i in range(args.warmup):
        cpu_oracle_rows(inp, [int(order[(i * nrow + k) % nrows_all]) for k in range(nrow)])
    total_t, total_b = 0.0, 0.0
    for i in range(args.steps):
        sel = [int(order[(i * nrow + k) % nrows_all]) for k in range(nrow)]
        t, b = cpu_oracle_rows(inp, sel)
        total_t += t
        total_b += b
    value = total_b / total_t / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": config_dict(cfg, inp, extra={"variant": variant_note(args.variant, args)}),
        "measurement": {"sample_rows_per_step": nrow, "timing": "host wall clock per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{nrow} of {nrows_all} output rows (query heads of sequences) per step, "
                                   f"seeded order, float64 oracle (OpenMP over rows)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_meanpool(args) -> None:
    """The fp32 mean-pool oracle as the reference arm: one whole conversion per step."""
    import oracle
    name, shp = meanpool_workload(args.workload or MEANPOOL_DEFAULT)
    H, G, h, dm, outer = shp["H"], shp["G"], shp["h"], shp["d_model"], shp.get("outer", 1)
    # one projection per step (the checkpoint's projections are independent conversions)
    w_h = make_meanpool_input(H, G, h, dm, shp["config_id"])
    alg = w_h.nbytes + G * h * dm * 4
    for _ in range(args.warmup):
        oracle.meanpool_f32(w_h, H, G)
    total_t = 0.0
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.meanpool_f32(w_h, H, G)
        total_t += time.perf_counter() - t
    value = args.steps * alg / total_t / 1e9
    sample = ("one whole conversion per step, fp32 oracle (one thread)" if outer == 1 else
              f"one [{H}, {h}, {dm}] projection of the {outer} per step, fp32 oracle (one thread)")
    line = {
        "metric": MEANPOOL_METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "reference",
        "config": {"workload": name, "H": H, "G": G, "h": h, "d_model": dm, "outer": outer,
                   "bytes_per_step": alg * outer},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank runs its own replica, the job ends with the last."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(kv_bytes_per_step: int, steps: int, world: int, total_ms: float) -> float:
    """Algorithmic KV bytes of all ranks' steps over the slowest rank's time (weak scaling)."""
    return world * kv_bytes_per_step * steps / (total_ms / 1e3) / 1e9


def variant_note(variant, args):
    return {"contiguous": "contiguous cache [B,G,Lmax,d]",
            "paged": f"paged cache, {args.page_size}-position pages in random pool order",
            "append": "fused append of the new token's K/V rows at position seq_lens[b]-1, then decode",
            "cross": "cross-attention: seq_lens NULL, all Lmax positions valid",
            "window": f"sliding window of the last {args.window} positions"}[variant]


def config_dict(cfg, inp, extra=None):
    """The workload's definition (the same keys and values in both arms' lines)."""
    d = {"workload": cfg.name, "B": cfg.B, "H": cfg.H, "G": cfg.G, "d": cfg.d, "Lmax": cfg.Lmax,
         "seq_lens": (list(cfg.fixed_seq) if cfg.fixed_seq else f"U[{cfg.seq_lo},{cfg.seq_hi}] seeded"),
         "kv_bytes_per_step": inp.kv_bytes, "inputs": "N(0,1) -> bf16, seeded",
         "l2": "inputs larger than L2: no step finds its K/V cache in L2"}
    if extra:
        d.update(extra)
    return d


def time_blocks(torch, dist, run_block, stream, world, dev, repeat_seconds, local_rank, clocks=True):
    """Times R back-to-back blocks (run_block(r) enqueues block r on `stream`), each between its own
    pair of CUDA events, with nvidia-smi clock samples during them; R is chosen from a first block so
    that they take about `repeat_seconds`.  Returns (median block ms, max over ranks), the sorted
    block times, R and the clock summary."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run_block(0)
    e1.record(stream)
    torch.cuda.synchronize()
    est = max(float(e0.elapsed_time(e1)), 1e-3)
    R = int(min(20000, max(3, math.ceil(repeat_seconds * 1e3 / est))))
    if world > 1:   # every rank runs the same number of blocks
        t = torch.tensor([R], dtype=torch.int64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        R = int(t.item())
        dist.barrier()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(R)]
    with (ClockSampler(local_rank) if clocks else contextlib.nullcontext()) as clk:
        for r, (a, b) in enumerate(evs):
            a.record(stream)
            run_block(r + 1)
            b.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    blocks = sorted(float(a.elapsed_time(b)) for a, b in evs)
    med = max_over_ranks(statistics.median(blocks), world, dev)
    return med, blocks, R, (clk.summary() if clocks else None)


def block_stats(blocks, R, steps):
    return {"blocks": R, "steps_per_block": steps, "median_ms": statistics.median(blocks),
            "p10_ms": blocks[int(0.1 * (len(blocks) - 1))], "p90_ms": blocks[int(0.9 * (len(blocks) - 1))]}


def make_graphs(torch, step, stream, K, period):
    """CUDA graphs of K steps (step(i) enqueues step i through the public API on the current stream),
    one for each starting offset of the copy schedule (i mod period), so that consecutive blocks
    continue the schedule; None if capture is not available."""
    offsets = []
    o = 0
    while o not in offsets:
        offsets.append(o)
        o = (o + K) % period
    graphs = {}
    try:
        for o in offsets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(K):
                    step(o + i)
            graphs[o] = g
    except RuntimeError:
        return None, offsets
    return graphs, offsets


def block_runner(torch, step, stream, K, period):
    """run_block(r): block r of K steps, as a graph replay (or K eager calls if capture fails)."""
    graphs, offsets = make_graphs(torch, step, stream, K, period)

    def run_block(r):
        o = offsets[r % len(offsets)]
        if graphs is not None:
            graphs[o].replay()
        else:
            for i in range(K):
                step(o + i)

    with torch.cuda.stream(stream):   # warm the graphs (and the eager path's host side)
        for r in range(len(offsets)):
            run_block(r)
    torch.cuda.synchronize()
    return run_block, graphs is not None


def run_meanpool(args, world, rank, local_rank, dev, torch, dist, gqa) -> None:
    """Times the mean-pool conversion, one call per step: one projection [H, h, d_model] fp32 ->
    [G, h, d_model] (gqa_meanpool_kv), or a whole checkpoint [outer, H, h*d_model] ->
    [outer, G, h*d_model] in one strided call (gqa_meanpool_kv_strided)."""
    name, shp = meanpool_workload(args.workload or MEANPOOL_DEFAULT)
    H, G, h, dm, outer = shp["H"], shp["G"], shp["h"], shp["d_model"], shp.get("outer", 1)
    w_h = make_meanpool_input(H, G, h, dm, shp["config_id"], outer=outer)
    in_bytes, out_bytes = w_h.nbytes, outer * G * h * dm * 4
    alg = in_bytes + out_bytes                  # each input read once, each output written once
    out_shape = (G, h, dm) if outer == 1 else (outer, G, h * dm)
    stream = torch.cuda.Stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = 2 if alg > 8 * l2 else max(3, math.ceil(L2_COPIES_SPAN * l2 / alg) + 1)
    w = torch.from_numpy(w_h).to(dev)
    ws = [w] + [w.clone() for _ in range(copies - 1)]
    outs = [torch.empty(out_shape, dtype=torch.float32, device=dev) for _ in range(copies)]
    convert = gqa.meanpool_kv if outer == 1 else gqa.meanpool_kv_strided

    def step(i):
        c = i % copies
        convert(ws[c], G, out=outs[c], stream=torch.cuda.current_stream(dev))

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize()
    run_block, graphed = block_runner(torch, step, stream, args.steps, copies)
    with torch.cuda.stream(stream):
        med_ms, blocks, R, clocks = time_blocks(torch, dist, run_block, stream, world, dev, args.repeat_seconds,
                                                local_rank)
    ms_per_step = med_ms / args.steps
    value = whole_job_gbs(alg, args.steps, world, med_ms)
    del ws[1:]
    torch.cuda.empty_cache()

    hw = torch.from_numpy(w_h).pin_memory()
    hout = torch.empty(out_shape, dtype=torch.float32).pin_memory()
    cur = torch.cuda.current_stream(dev)
    e2e_steps = args.e2e_steps if in_bytes < (1 << 30) else min(args.e2e_steps, 3)

    def e2e_step():
        w.copy_(hw, non_blocking=True)
        convert(w, G, out=outs[0], stream=cur)
        hout.copy_(outs[0], non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(cur)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    if rank != 0:
        return

    peak, peak_kind = measured_peak()
    achieved = alg / (ms_per_step / 1e3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        one = w_h if outer == 1 else w_h[0].reshape(H, h, dm)   # one projection: a bounded sample
        one_bytes = one.nbytes + G * h * dm * 4
        oracle.meanpool_f32(one, H, G)               # warm: page faults
        total_t, passes = 0.0, 0
        while total_t < CPU_BASELINE_SECONDS / 4 and passes < 10000:
            t = time.perf_counter()
            oracle.meanpool_f32(one, H, G)
            total_t += time.perf_counter() - t
            passes += 1
        cpu = {"value": passes * one_bytes / total_t / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{passes} conversion(s) of one [{H}, {h}, {dm}] projection"
                         + ("" if outer == 1 else f" (of the {outer})")
                         + f", fp32 oracle (one thread), {total_t:.1f} s after one warm-up pass"}
    layout = ("[H, h, d_model] -> [G, h, d_model] fp32, head-major" if outer == 1 else
              f"[{outer}, H, h*d_model] -> [{outer}, G, h*d_model] fp32: every K and V projection of the "
              f"checkpoint in one strided call")
    line = {
        "metric": MEANPOOL_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": name, "H": H, "G": G, "h": h, "d_model": dm, "outer": outer,
                   "layout": layout, "bytes_per_step": alg, "inputs": "N(0,1) float32, seeded",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU", "copies": copies,
                   "l2": f"inputs larger than L2: {copies} input/output copies, step i uses copy i % {copies}"
                         if copies * alg > l2 else "fits in L2: launch-bound, not an HBM figure",
                   "timing": ("median of R blocks of K calls, each block a CUDA-graph replay between its own "
                              "pair of CUDA events" if graphed else "median of R blocks of K eager calls")},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": profiled_traffic("meanpool_kernel", name), "kernel": "meanpool_kernel",
                     "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
                     "algorithmic_bytes_per_launch": alg, "frac_of_8TBps_nominal": achieved / 8000.0},
        "cpu_baseline": cpu,
        "e2e": {"value": alg / (e2e_ms / 1e3) / 1e9 * world, "unit": UNIT, "h2d_bytes_per_step": in_bytes,
                "d2h_bytes_per_step": out_bytes, "steps": e2e_steps,
                "what": "H2D of the projections from pinned host memory + the conversion + D2H of the result"},
        "timing": block_stats(blocks, R, args.steps),
        "gpu_launches": args.steps * R,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


READONLY_SHAPE = (1024, 8192)   # [z, rows] of 256-byte rows: 2 GiB, 17x the L2


def measure_readonly(torch, dist, gqa, dev, world, local_rank, repeat_seconds):
    """The read-bandwidth ceiling: GB/s of the read-only TMA stream (gqa_bench.h) over a 2 GiB buffer,
    median of R calls, each between its own pair of CUDA events."""
    z, rows = READONLY_SHAPE
    buf = torch.empty((z, rows, 128), dtype=torch.bfloat16, device=dev)
    buf.view(torch.int16).fill_(0x3F80)    # bf16 1.0: the data is never used, only read
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    nbytes = buf.numel() * 2

    def run_block(r):
        gqa.stream_read(buf, flags, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            run_block(0)
    torch.cuda.synchronize()
    med_ms, blocks, R, clocks = time_blocks(torch, dist, run_block, stream, world, dev, repeat_seconds, local_rank)
    torch.cuda.synchronize()
    if int(flags.item()) != 0:
        raise RuntimeError(f"read-only stream reported flags 0x{int(flags.item()):x}")
    del buf
    return {"value": nbytes / (med_ms / 1e3) / 1e9, "best": nbytes / (blocks[0] / 1e3) / 1e9, "unit": UNIT,
            "bytes_per_call": nbytes, "calls": R, "clocks": clocks,
            "what": "read-only TMA stream, one CTA per SM, the decode's 64-column x 128-row boxes (two per 32 KiB "
                    "tile), six-stage ring, 2 GiB buffer; median of R calls"}


PAGE_SWEEP = (   # (page rows, boxes per page, issuing warps, lanes per warp)
    [(r, 2, 1, l) for r in (16, 32, 64, 128) for l in (1, 2, 4, 8, 16) if l <= 256 // r] +
    [(r, 1, 1, l) for r in (16, 32, 64) for l in (1, 2, 4, 8) if l <= 128 // r] +
    [(16, 2, 2, 16), (16, 1, 2, 1), (16, 1, 2, 8)])


def measure_page_boxes(torch, dist, gqa, dev, world, local_rank, repeat_seconds):
    """The per-box cost of small pages: GB/s of the read-only stream when every 32 KiB tile is
    fetched as pages of 16..128 rows at scattered places of a 2 GiB pool, two boxes per page (the
    whole-tile layout) or one (a five-dimensional tensor map), issued by L lanes of one or two warps
    per SM (gqa_bench_stream_read_pages); median of R calls each."""
    z, rows = READONLY_SHAPE
    buf = torch.empty((z, rows, 128), dtype=torch.bfloat16, device=dev)
    buf.view(torch.int16).fill_(0x3F80)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    nbytes = buf.numel() * 2
    table = []
    for pr, per_page, warps, lanes in PAGE_SWEEP:
        def run_block(r, pr=pr, lanes=lanes, one=per_page == 1, warps=warps):
            gqa.stream_read_pages(buf, flags, pr, lanes, scatter=True, one_box=one, warps=warps, stream=stream)

        try:
            with torch.cuda.stream(stream):
                for _ in range(3):
                    run_block(0)
        except gqa.GQAError as e:   # the driver may refuse a map: report it, run the rest
            table.append({"page_rows": pr, "boxes_per_page": per_page, "warps": warps, "lanes": lanes,
                          "error": str(e)})
            continue
        torch.cuda.synchronize()
        med_ms, blocks, R, _ = time_blocks(torch, dist, run_block, stream, world, dev, repeat_seconds,
                                           local_rank, clocks=False)
        gbs = nbytes / (med_ms / 1e3) / 1e9
        boxes = (128 // pr) * per_page
        table.append({"page_rows": pr, "boxes_per_page": per_page, "warps": warps, "lanes": lanes,
                      "gbs": round(gbs, 1), "ns_per_box_per_sm": round(32768 / boxes / (gbs / 148), 2)})
    torch.cuda.synchronize()
    if int(flags.item()) != 0:
        raise RuntimeError(f"paged read-only stream reported flags 0x{int(flags.item()):x}")
    del buf
    return {"unit": UNIT, "bytes_per_call": nbytes,
            "what": "read-only TMA stream over a 2 GiB pool read as pages of R rows (R x 256 bytes) at scattered "
                    "places, a 32 KiB tile = 128/R pages, two 64-column boxes per page or one five-dimensional box, "
                    "issued by L lanes of W warps per SM (W warps take alternate tiles); GB/s and the time per box "
                    "per SM it implies (median of R calls)",
            "sweep": table}


def decode_case(args, cfg, variant, torch, gqa, dev):
    """Inputs, cache copies, workspace and the step function of one decode workload on the device."""
    if variant == "cross":   # every one of the Lmax positions is valid
        inp = make_decode_inputs(cfg, poison_tail=False, seq_lens=[cfg.Lmax] * cfg.B)
    else:
        inp = make_decode_inputs(cfg, poison_tail=False)
    window = args.window if variant == "window" else 0
    attended = np.minimum(inp.seq_lens.astype(np.int64), window) if window else inp.seq_lens.astype(np.int64)
    kv_bytes = int(attended.sum()) * cfg.G * cfg.d * 2 * 2   # algorithmic K+V bytes of one step
    scale = float(inp.scale)
    path = args.path or gqa.select_path(cfg.B, cfg.H, cfg.G, cfg.d, cfg.Lmax)
    if variant != "contiguous" and path != gqa.PATH_TCGEN05:
        raise SystemExit("the decode variants run on the tensor-core path")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def to_dev(a, dtype=torch.bfloat16):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(dtype) if dtype == torch.bfloat16 else t).to(dev)

    q = to_dev(inp.q)
    sl = to_dev(inp.seq_lens, torch.int32)
    kn = vn = kn_h = vn_h = None
    if variant == "paged":
        kp, vp, table = make_paged_layout(inp, args.page_size)
        k, v, tbl = to_dev(kp), to_dev(vp), to_dev(table, torch.int32)
        host_kv = (kp, vp, table)
    else:
        k, v, tbl = to_dev(inp.k), to_dev(inp.v), None
        host_kv = (inp.k, inp.v)
    if variant == "append":
        kn_h, vn_h = make_new_rows(cfg)
        kn, vn = to_dev(kn_h), to_dev(vn_h)
    copies = max(3, math.ceil(L2_COPIES_SPAN * l2 / kv_bytes) + 1)
    ks = [k] + [k.clone() for _ in range(copies - 1)]
    vs = [v] + [v.clone() for _ in range(copies - 1)]
    out = torch.empty((cfg.B, cfg.H, cfg.d), dtype=torch.float32, device=dev)
    ws = gqa.alloc_workspace(cfg.B, cfg.H, cfg.G, cfg.d, cfg.Lmax, dev)

    def call(kk, vv):
        st = torch.cuda.current_stream(dev)
        if variant == "paged":
            gqa.decode_paged(q, kk, vv, tbl, sl, out=out, workspace=ws, scale=scale, stream=st)
        elif variant == "append":
            gqa.decode_append(q, kn, vn, kk, vv, sl, out=out, workspace=ws, scale=scale, stream=st)
        else:
            gqa.decode(q, kk, vv, None if variant == "cross" else sl, out=out, workspace=ws, scale=scale,
                       stream=st, path=path, window=window)

    def step(i):
        c = i % copies
        call(ks[c], vs[c])

    return dict(inp=inp, kv_bytes=kv_bytes, path=path, copies=copies, step=step, call=call, q=q, sl=sl, k=k, v=v,
                tbl=tbl, kn=kn, vn=vn, kn_h=kn_h, vn_h=vn_h, host_kv=host_kv, out=out, ws=ws, window=window)


def measure_decode(args, cfg, variant, world, local_rank, dev, torch, dist, gqa, e2e=True):
    """The timed step of one decode workload (see the module docstring) and its end-to-end figure."""
    c = decode_case(args, cfg, variant, torch, gqa, dev)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            c["step"](i)
    torch.cuda.synchronize()
    run_block, graphed = block_runner(torch, c["step"], stream, args.steps, c["copies"])
    with torch.cuda.stream(stream):
        med_ms, blocks, R, clocks = time_blocks(torch, dist, run_block, stream, world, dev, args.repeat_seconds,
                                                local_rank)
    flags = gqa.read_flags(c["ws"])
    if flags:
        raise RuntimeError(f"decode reported flags 0x{flags:x} during the benchmark")
    res = {"cfg": cfg, "inp": c["inp"], "kv_bytes": c["kv_bytes"], "path": c["path"], "copies": c["copies"],
           "ms_per_step": med_ms / args.steps, "value": whole_job_gbs(c["kv_bytes"], args.steps, world, med_ms),
           "timing": block_stats(blocks, R, args.steps), "R": R, "clocks": clocks, "graphed": graphed,
           "window": c["window"]}
    if e2e:
        res["e2e"] = measure_e2e(args, c, variant, world, dev, torch)
    return res


def measure_e2e(args, c, variant, world, dev, torch):
    """The same metric through the public API with host buffers: every step copies all of its inputs
    from pinned host memory (the whole caches or page pools included), decodes, and reads out back."""
    def pinned(a, dtype=torch.bfloat16):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(dtype) if dtype == torch.bfloat16 else t).pin_memory()

    inp = c["inp"]
    host = [(c["q"], pinned(inp.q)), (c["sl"], pinned(inp.seq_lens, torch.int32)), (c["k"], pinned(c["host_kv"][0])),
            (c["v"], pinned(c["host_kv"][1]))]
    if c["tbl"] is not None:
        host.append((c["tbl"], pinned(c["host_kv"][2], torch.int32)))
    if variant == "append":
        host += [(c["kn"], pinned(c["kn_h"])), (c["vn"], pinned(c["vn_h"]))]
    out = c["out"]
    hout = torch.empty(tuple(out.shape), dtype=torch.float32).pin_memory()
    h2d = sum(h.numel() * h.element_size() for _, h in host)
    d2h = hout.numel() * 4
    cur = torch.cuda.current_stream(dev)

    def e2e_step():
        for dst, src in host:
            dst.copy_(src, non_blocking=True)
        c["call"](c["k"], c["v"])
        hout.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(cur)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, world, dev)
    return {"value": whole_job_gbs(c["kv_bytes"], 1, world, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
            "what": "H2D of every input (q, seq_lens, the whole K/V caches or page pools, the block table and "
                    "appended rows where used) from pinned host memory + the decode call + D2H of out, per step"}


def roofline_of(res, variant, readonly, kernel="gqa_decode_tc_kernel"):
    peak, peak_kind = measured_peak()
    achieved = res["kv_bytes"] / (res["ms_per_step"] / 1e3) / 1e9
    r = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
         "traffic": profiled_traffic(kernel, res["cfg"].name) if variant == "contiguous" else None,
         "kernel": kernel, "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind}, a copy)",
         "algorithmic_bytes_per_launch": res["kv_bytes"], "frac_of_8TBps_nominal": achieved / 8000.0,
         "achieved_covers": "whole steps (decode kernel + split-combine kernel)"}
    if readonly:
        r["readonly_peak"] = readonly["value"]
        r["frac_of_readonly"] = achieved / readonly["value"]
        r["readonly_peak_source"] = "measured in this run: gqa_bench_stream_read (read-only TMA stream)"
    return r


def cpu_baseline_decode(inp, window):
    """The float64 oracle on the host cores (all of them, then one thread), each on a bounded sample of
    the workload's (batch, K/V head) segments."""
    import oracle
    cfg = inp.cfg
    segs = all_segments(cfg)

    def sample(seconds):
        cpu_oracle_step(inp, segs[:1], window)               # warm: thread pool, page faults
        t, _ = cpu_oracle_step(inp, segs[:1], window)
        nseg = int(max(1, min(len(segs), seconds / max(t, 1e-4))))
        total_t, total_b, passes = 0.0, 0, 0
        while total_t < seconds and passes < 1000:
            t, b = cpu_oracle_step(inp, segs[:nseg], window)
            total_t += t
            total_b += b
            passes += 1
        return total_b / total_t / 1e9, nseg, passes, total_t

    cores = oracle.num_threads()
    v, nseg, passes, tt = sample(CPU_BASELINE_SECONDS)
    oracle.set_num_threads(1)
    try:
        v1, nseg1, passes1, tt1 = sample(CPU_BASELINE_SECONDS / 2)
    finally:
        oracle.set_num_threads(cores)
    return {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{passes} pass(es) over {nseg} of {len(segs)} (batch, K/V head) segments, all H/G query "
                      f"heads each, float64 oracle, {tt:.1f} s after one warm-up pass",
            "cores_1": {"value": v1, "unit": UNIT, "cores": 1,
                        "sample": f"{passes1} pass(es) over {nseg1} segments, one thread, {tt1:.1f} s"}}


def run_readonly(args, world, rank, local_rank, dev, torch, dist, gqa) -> None:
    """--variant readonly: the read-only stream's own line."""
    ro = measure_readonly(torch, dist, gqa, dev, world, local_rank, args.repeat_seconds)
    pages = measure_page_boxes(torch, dist, gqa, dev, world, local_rank, min(args.repeat_seconds, 0.15))
    if rank != 0:
        return
    peak, peak_kind = measured_peak()
    line = {"metric": "read-only TMA stream GB/s (the decode's read ceiling), 1 GPU", "value": ro["value"] * world,
            "unit": UNIT, "n_gpus": world, "steps": ro["calls"], "warmup": 3,
            "ms_per_step": ro["bytes_per_call"] / ro["value"] / 1e6, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "readonly_stream", "bytes_per_step": ro["bytes_per_call"], "what": ro["what"]},
            "roofline": {"bound": "hbm", "achieved": ro["value"], "peak": peak, "unit": "GB/s",
                         "frac": ro["value"] / peak, "traffic": None, "kernel": "stream_read_kernel",
                         "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind}, a copy)"},
            "best": ro["best"], "gpu_launches": ro["calls"], "clocks": ro["clocks"], "page_boxes": pages}
    print(json.dumps(line), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=None,
                    help="llama3_70b (default) | mistral7b | long_ragged | tiny | t5xxl_sweep_G<1..64>; "
                         "--variant meanpool: t5xxl_checkpoint (default) | tiny | t5xxl_sweep_G<g>")
    ap.add_argument("--secondary", default="mistral7b",
                    help="a second workload measured in the same run and reported in the line's 'secondary' "
                         "object (contiguous cache only; 'none' to skip)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", type=int, default=0, help="0 auto, 1 simt, 2 tcgen05")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--repeat-seconds", type=float, default=1.5,
                    help="about how long the repeated timed blocks of a workload take (clock samples)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-readonly", action="store_true", help="skip the read-only ceiling measurement")
    ap.add_argument("--variant", default="contiguous",
                    choices=["contiguous", "paged", "append", "cross", "window", "meanpool", "readonly"],
                    help="contiguous cache (default); paged cache (--page-size); fused append of the new "
                         "token's K/V rows; cross-attention (every position valid); sliding window (--window); "
                         "meanpool: the K/V mean-pool conversion instead of the decode; readonly: the read-only "
                         "stream that bounds the decode")
    ap.add_argument("--page-size", type=int, default=64)
    ap.add_argument("--window", type=int, default=1024)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    import torch.distributed as dist
    from kv_cache_decode_06_b300 import build_lib, gqa

    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    build_lib.build()
    build_lib.build(bench=True)
    gqa.load()
    try:
        if args.variant == "meanpool":
            run_meanpool(args, world, rank, local_rank, dev, torch, dist, gqa)
        elif args.variant == "readonly":
            run_readonly(args, world, rank, local_rank, dev, torch, dist, gqa)
        else:
            run_decode(args, world, rank, local_rank, dev, torch, dist, gqa)
    finally:
        if world > 1:
            dist.destroy_process_group()


def run_decode(args, world, rank, local_rank, dev, torch, dist, gqa) -> None:
    variant = args.variant
    cfg = workload(args.workload or "llama3_70b")
    prim = measure_decode(args, cfg, variant, world, local_rank, dev, torch, dist, gqa)
    torch.cuda.empty_cache()
    sec = None
    if args.secondary != "none" and variant == "contiguous" and args.secondary != cfg.name:
        sec = measure_decode(args, workload(args.secondary), "contiguous", world, local_rank, dev, torch, dist, gqa,
                             e2e=False)
        torch.cuda.empty_cache()
    readonly = None if args.no_readonly else measure_readonly(torch, dist, gqa, dev, world, local_rank,
                                                             min(args.repeat_seconds, 0.5))
    if rank != 0:
        return
    kernel = "gqa_decode_tc_kernel" if prim["path"] == gqa.PATH_TCGEN05 else "gqa_decode_simt_kernel"
    cpu = None if args.no_cpu_baseline else cpu_baseline_decode(prim["inp"], prim["window"])
    timing = ("K steps captured in CUDA graphs (public API calls); the median of R blocks, each one graph "
              "replay between its own pair of CUDA events" if prim["graphed"] else
              "the median of R blocks of K eager steps, each between its own pair of CUDA events")
    line = {
        "metric": METRIC, "value": prim["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": prim["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if prim["path"] == gqa.PATH_TCGEN05 else "f32", "data": "synthetic",
        "steps_per_s": world * 1e3 / prim["ms_per_step"],
        "config": config_dict(cfg, prim["inp"], extra={"variant": variant_note(variant, args)}),
        "measurement": {
            "path": "tcgen05" if prim["path"] == gqa.PATH_TCGEN05 else "simt",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU", "cache_copies": prim["copies"],
            "l2": f"K/V caches held in {prim['copies']} copies, step i reads copy i % {prim['copies']}, so >= "
                  f"{L2_COPIES_SPAN} L2 capacities of other KV data stream between two reads of a copy",
            "timing": timing},
        "roofline": roofline_of(prim, variant, readonly, kernel),
        "cpu_baseline": cpu,
        "e2e": prim["e2e"],
        "timing": prim["timing"],
        "gpu_launches": 2 * args.steps * prim["R"],   # decode + split-combine per step, every timed block
        "clocks": prim["clocks"],
    }
    if sec is not None:
        line["secondary"] = {
            "workload": sec["cfg"].name, "value": sec["value"], "unit": UNIT, "ms_per_step": sec["ms_per_step"],
            "steps_per_s": world * 1e3 / sec["ms_per_step"],
            "config": config_dict(sec["cfg"], sec["inp"], extra={"variant": variant_note("contiguous", args)}),
            "cache_copies": sec["copies"],
            "roofline": roofline_of(sec, "contiguous", readonly, kernel), "timing": sec["timing"],
            "gpu_launches": 2 * args.steps * sec["R"], "clocks": sec["clocks"]}
    if readonly is not None:
        line["readonly_stream"] = {k: readonly[k] for k in ("value", "best", "unit", "bytes_per_call", "calls",
                                                             "what")}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
