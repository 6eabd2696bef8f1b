"""Benchmark of one GQA decode step (KV-cache HBM GB/s and decode steps/s).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one gqa_decode call on the workload's whole batch (one layer), with
the bf16 KV cache resident in HBM.  GB/s counts algorithmic bytes only: the
valid K and V rows, sum_b seq_lens[b] * G * d * 2 bytes * 2.

L2: inputs larger than L2.  The K/V caches are held in C copies and step i
reads copy i % C, with C chosen so that the C - 1 steps between two reads of a
copy stream at least three L2 capacities of other data; no step finds its
cache in L2.  (A write-flush between steps is not used: the dirty lines it
leaves slow the next kernel down by write-back traffic that is not its own.)
The K steps run back to back on one stream between one pair of CUDA events;
a step is the decode kernel plus the split-combine kernel that follows it
(programmatic dependent launch), so total time / K is the average duration of
one whole step.

``--variant meanpool`` times the K/V mean-pool conversion instead (one call per
step on one projection; GB/s counts its input and output bytes).

Under torchrun (N > 1) every rank runs an independent replica of the step on
its own GPU (nothing is sharded); value = bytes of all ranks / max time.

``--impl reference`` times the float64 CPU oracle on the host cores instead, on
a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
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
    CONFIGS, MEANPOOL_T5XXL, MEANPOOL_TINY, T5XXL_SWEEP_GS, make_decode_inputs, make_meanpool_input,
    make_new_rows, make_paged_layout,
)

METRIC = "GQA decode KV-cache HBM GB/s (% of B300 peak) and decode steps/s, 1 GPU"
MEANPOOL_METRIC = "GQA K/V mean-pool conversion HBM GB/s (% of B300 peak), 1 GPU"
UNIT = "GB/s"
L2_COPIES_SPAN = 3            # L2 capacities streamed between two reads of one cache copy
CPU_BASELINE_SECONDS = 10.0   # host time spent on the float64 oracle for the cpu_baseline field
FALLBACK_HBM_GBS = 6400.0


def meanpool_workload(name: str):
    """Shape of one mean-pool conversion (one projection of one layer)."""
    if name == "tiny":
        return "meanpool_tiny", dict(MEANPOOL_TINY)
    if name.startswith("t5xxl_sweep_G"):
        d = dict(MEANPOOL_T5XXL)
        d["G"] = int(name.split("_G")[1])
        return f"meanpool_t5xxl_G{d['G']}", d
    raise SystemExit(f"--variant meanpool takes --workload tiny or t5xxl_sweep_G<g>, not {name}")


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
    cfg = workload(args.workload or "mistral7b")
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
        "config": config_dict(cfg, inp, extra={"sample_rows_per_step": nrow}),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{nrow} of {nrows_all} output rows (query heads of sequences) per step, "
                                   f"seeded order, float64 oracle (OpenMP over rows)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_meanpool(args) -> None:
    """The fp32 mean-pool oracle as the reference arm: one whole conversion per step."""
    import oracle
    name, shp = meanpool_workload(args.workload or "t5xxl_sweep_G8")
    H, G, h, dm = shp["H"], shp["G"], shp["h"], shp["d_model"]
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
    line = {
        "metric": MEANPOOL_METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "reference",
        "config": {"workload": name, "H": H, "G": G, "h": h, "d_model": dm, "bytes_per_step": alg},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "one whole conversion per step, fp32 oracle (one thread)"},
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
    d = {"workload": cfg.name, "B": cfg.B, "H": cfg.H, "G": cfg.G, "d": cfg.d, "Lmax": cfg.Lmax,
         "seq_lens": (list(cfg.fixed_seq) if cfg.fixed_seq else f"U[{cfg.seq_lo},{cfg.seq_hi}] seeded"),
         "kv_bytes_per_step": inp.kv_bytes, "inputs": "N(0,1) -> bf16, seeded",
         "l2": "inputs larger than L2: no step finds its K/V cache in L2"}
    if extra:
        d.update(extra)
    return d


def run_meanpool(args, world, rank, local_rank, dev, torch, dist, gqa) -> None:
    """Times gqa_meanpool_kv: [H, h, d_model] fp32 -> [G, h, d_model] fp32, one call per step."""
    name, shp = meanpool_workload(args.workload or "t5xxl_sweep_G8")
    H, G, h, dm = shp["H"], shp["G"], shp["h"], shp["d_model"]
    w_h = make_meanpool_input(H, G, h, dm, shp["config_id"])
    in_bytes, out_bytes = w_h.nbytes, G * h * dm * 4
    alg = in_bytes + out_bytes                  # each input read once, each output written once
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = max(3, math.ceil(L2_COPIES_SPAN * l2 / alg) + 1)
    w = torch.from_numpy(w_h).to(dev)
    ws = [w] + [w.clone() for _ in range(copies - 1)]
    outs = [torch.empty((G, h, dm), dtype=torch.float32, device=dev) for _ in range(copies)]

    def step(i):
        c = i % copies
        gqa.meanpool_kv(ws[c], G, out=outs[c], stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t0.record(stream)
        for i in range(args.steps):
            step(i)
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms = max_over_ranks(float(t0.elapsed_time(t1)), world, dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_gbs(alg, args.steps, world, total_ms)

    hw = torch.from_numpy(w_h).pin_memory()
    hout = torch.empty((G, h, dm), dtype=torch.float32).pin_memory()

    def e2e_step():
        w.copy_(hw, non_blocking=True)
        gqa.meanpool_kv(w, G, out=outs[0], stream=stream)
        hout.copy_(outs[0], non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, world, dev)
    if rank != 0:
        return

    peak, peak_kind = measured_peak()
    achieved = alg / (ms_per_step / 1e3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        oracle.meanpool_f32(w_h, H, G)               # warm: page faults
        total_t, passes = 0.0, 0
        while total_t < CPU_BASELINE_SECONDS / 4 and passes < 10000:
            t = time.perf_counter()
            oracle.meanpool_f32(w_h, H, G)
            total_t += time.perf_counter() - t
            passes += 1
        cpu = {"value": passes * alg / total_t / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{passes} whole conversion(s) of the same projection, fp32 oracle (one thread), "
                         f"{total_t:.1f} s after one warm-up pass"}
    line = {
        "metric": MEANPOOL_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": name, "H": H, "G": G, "h": h, "d_model": dm,
                   "layout": "[H, h, d_model] -> [G, h, d_model] fp32, head-major",
                   "bytes_per_step": alg, "inputs": "N(0,1) float32, seeded",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU", "copies": copies,
                   "l2": f"inputs larger than L2: {copies} input/output copies, step i uses copy i % {copies}"
                         if copies * alg > l2 else "fits in L2: launch-bound, not an HBM figure",
                   "timing": "K calls back to back between one pair of CUDA events"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": profiled_traffic("meanpool_kernel", name), "kernel": "meanpool_kernel",
                     "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
                     "algorithmic_bytes_per_launch": alg, "frac_of_8TBps_nominal": achieved / 8000.0},
        "cpu_baseline": cpu,
        "e2e": {"value": alg / (e2e_ms / 1e3) / 1e9 * world, "unit": UNIT, "h2d_bytes_per_step": in_bytes,
                "d2h_bytes_per_step": out_bytes, "steps": args.e2e_steps,
                "what": "H2D of the projection from pinned host memory + the conversion + D2H of the result"},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default=None,
                    help="mistral7b (default) | llama3_70b | long_ragged | tiny | t5xxl_sweep_G<1..64>; "
                         "--variant meanpool: tiny | t5xxl_sweep_G<g> (default t5xxl_sweep_G8)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", type=int, default=0, help="0 auto, 1 simt, 2 tcgen05")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--variant", default="contiguous",
                    choices=["contiguous", "paged", "append", "cross", "window", "meanpool"],
                    help="contiguous cache (default); paged cache (--page-size); fused append of the new "
                         "token's K/V rows; cross-attention (every position valid); sliding window (--window); "
                         "meanpool: the K/V mean-pool conversion instead of the decode")
    ap.add_argument("--page-size", type=int, default=64)
    ap.add_argument("--window", type=int, default=1024)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

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
    gqa.load()
    if args.variant == "meanpool":
        run_meanpool(args, world, rank, local_rank, dev, torch, dist, gqa)
        if world > 1:
            dist.destroy_process_group()
        return

    cfg = workload(args.workload or "mistral7b")
    variant = args.variant
    if variant == "cross":   # every one of the Lmax positions is valid
        inp = make_decode_inputs(cfg, poison_tail=False, seq_lens=[cfg.Lmax] * cfg.B)
    else:
        inp = make_decode_inputs(cfg, poison_tail=False)
    window = args.window if variant == "window" else 0
    attended = np.minimum(inp.seq_lens.astype(np.int64), window) if window else inp.seq_lens.astype(np.int64)
    kv_bytes = int(attended.sum()) * cfg.G * cfg.d * 2 * 2   # algorithmic K+V bytes of one step
    stream = torch.cuda.current_stream(dev)
    scale = float(inp.scale)
    path = args.path or gqa.select_path(cfg.B, cfg.H, cfg.G, cfg.d, cfg.Lmax)
    if variant != "contiguous" and path != gqa.PATH_TCGEN05:
        ap.error("the decode variants run on the tensor-core path")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def to_dev(a, dtype=torch.bfloat16):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(dtype) if dtype == torch.bfloat16 else t).to(dev)

    q = to_dev(inp.q)
    sl = to_dev(inp.seq_lens, torch.int32)
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
        if variant == "paged":
            gqa.decode_paged(q, kk, vv, tbl, sl, out=out, workspace=ws, scale=scale, stream=stream)
        elif variant == "append":
            gqa.decode_append(q, kn, vn, kk, vv, sl, out=out, workspace=ws, scale=scale, stream=stream)
        else:
            gqa.decode(q, kk, vv, None if variant == "cross" else sl, out=out, workspace=ws, scale=scale,
                       stream=stream, path=path, window=window)

    def step(i):
        c = i % copies
        call(ks[c], vs[c])

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t0.record(stream)
        for i in range(args.steps):
            step(i)
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms = max_over_ranks(float(t0.elapsed_time(t1)), world, dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_gbs(kv_bytes, args.steps, world, total_ms)
    flags = gqa.read_flags(ws)
    if flags:
        raise RuntimeError(f"decode reported flags 0x{flags:x} during the benchmark")

    # ---- per-step distribution (extra information): each of a few hundred steps between its own
    # pair of events; the events themselves serialise the steps, so this is not the headline number
    nper = min(200, args.steps)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nper)]
    for i, (ea, eb) in enumerate(evs):
        ea.record(stream)
        step(i)
        eb.record(stream)
    torch.cuda.synchronize()
    per_us = sorted(1e3 * ea.elapsed_time(eb) for ea, eb in evs)
    per_step = {"samples": nper, "median_us": statistics.median(per_us),
                "p10_us": per_us[int(0.1 * (nper - 1))], "p90_us": per_us[int(0.9 * (nper - 1))],
                "what": "each step alone between its own event pair: launch gaps included and no overlap "
                        "with the neighbouring steps (the headline times K steps back to back)"}

    # ---- end to end through the public API with host buffers (pinned)
    def pinned(a, dtype=torch.bfloat16):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(dtype) if dtype == torch.bfloat16 else t).pin_memory()

    host = [(q, pinned(inp.q)), (sl, pinned(inp.seq_lens, torch.int32)), (k, pinned(host_kv[0])),
            (v, pinned(host_kv[1]))]
    if tbl is not None:
        host.append((tbl, pinned(host_kv[2], torch.int32)))
    if variant == "append":
        host += [(kn, pinned(kn_h)), (vn, pinned(vn_h))]
    hout = torch.empty((cfg.B, cfg.H, cfg.d), dtype=torch.float32).pin_memory()
    h2d = sum(h.numel() * h.element_size() for _, h in host)
    d2h = hout.numel() * 4

    def e2e_step():
        for dst, src in host:
            dst.copy_(src, non_blocking=True)
        call(k, v)
        hout.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, world, dev)
    e2e_value = whole_job_gbs(kv_bytes, 1, world, e2e_ms)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peak()
    kernel = "gqa_decode_tc_kernel" if path == gqa.PATH_TCGEN05 else "gqa_decode_simt_kernel"
    achieved = kv_bytes / (ms_per_step / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": profiled_traffic(kernel, cfg.name) if variant == "contiguous" else None,
                "kernel": kernel,
                "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
                "algorithmic_bytes_per_launch": kv_bytes,
                "frac_of_8TBps_nominal": achieved / 8000.0}

    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        segs = all_segments(cfg)
        cpu_oracle_step(inp, segs[:1], window)               # warm: thread pool, page faults
        t, _ = cpu_oracle_step(inp, segs[:1], window)
        nseg = int(max(1, min(len(segs), CPU_BASELINE_SECONDS / max(t, 1e-4))))
        total_t, total_b, passes = 0.0, 0, 0
        while total_t < CPU_BASELINE_SECONDS and passes < 1000:
            t, b = cpu_oracle_step(inp, segs[:nseg], window)
            total_t += t
            total_b += b
            passes += 1
        cpu = {"value": total_b / total_t / 1e9, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{passes} pass(es) over {nseg} of {len(segs)} (batch, K/V head) segments, all H/G "
                         f"query heads each, float64 oracle, {total_t:.1f} s after one warm-up pass"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if path == gqa.PATH_TCGEN05 else "f32", "data": "synthetic",
        "steps_per_s": world * 1e3 / ms_per_step,
        "config": config_dict(cfg, inp, extra={"path": "tcgen05" if path == gqa.PATH_TCGEN05 else "simt",
                                               "variant": variant_note(variant, args),
                                               "kv_bytes_per_step": kv_bytes,
                                               "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                                               "cache_copies": copies,
                                               "l2": f"inputs larger than L2: K/V caches held in {copies} copies, "
                                                     f"step i reads copy i % {copies}, so >= {L2_COPIES_SPAN} L2 "
                                                     "capacities of other KV data stream between two reads of a copy",
                                               "timing": "K steps back to back between one pair of CUDA events"}),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": args.e2e_steps,
                "what": "H2D of every input (q, seq_lens, the whole K/V caches or page pools, the block table "
                        "and appended rows where used) from pinned host memory + the decode call + D2H of "
                        "out, per step"},
        "per_step_events": per_step,
        "gpu_launches": 2 * args.steps,   # decode kernel + split-combine kernel per step
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
