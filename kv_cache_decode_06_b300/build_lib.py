"""Build the CUDA library ``libgqa_b300.so`` in-tree with nvcc for sm_103a.

Usage: ``python -m kv_cache_decode_06_b300.build_lib [--force] [--verbose] [--trace] [--test-hooks] [--bench]``.
The shared library lands next to this file and is what the Python binding and
any C caller load.  ``-Xptxas -v`` output (registers, spills, shared memory) is
printed with ``--verbose``.  ``--trace`` builds ``libgqa_b300_trace.so`` instead:
the same library compiled with -DGQA_TRACE, whose tensor-core decode kernel
records a per-CTA timeline of its pipeline events (clock64 stamps) in a device
array that ``gqa_trace_copy(dst, bytes)`` copies to the host.  ``--test-hooks``
builds ``libgqa_b300_testhooks.so``: the same library compiled with
-DGQA_TEST_HOOKS, which also exports ``gqa_debug_withhold_copy`` (the failure-
path test's way to make a pipeline wait run out without a fault).  ``--bench``
builds ``libgqa_b300_bench.so`` from ``csrc_bench/`` (``include/gqa_bench.h``):
the read-only stream that measures the decode's read-bandwidth ceiling.
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libgqa_b300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
TRACE_LIB_PATH = os.path.join(HERE, "libgqa_b300_trace.so")
TEST_HOOKS_LIB_PATH = os.path.join(HERE, "libgqa_b300_testhooks.so")
BENCH_LIB_PATH = os.path.join(HERE, "libgqa_b300_bench.so")
CSRC_BENCH = os.path.join(HERE, "csrc_bench")
BUILD_DIR = os.path.join(HERE, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libgqa_b300.so")
    return cand


def sources(bench: bool = False):
    return sorted(glob.glob(os.path.join(CSRC_BENCH if bench else CSRC, "*.cu")))


def _stale(lib: str, bench: bool = False) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources(bench) + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]
    return any(os.path.getmtime(f) > t for f in deps)


def build(force: bool = False, verbose: bool = False, trace: bool = False, test_hooks: bool = False,
          bench: bool = False) -> str:
    if trace + test_hooks + bench > 1:
        raise ValueError("build one library variant at a time")
    lib = TRACE_LIB_PATH if trace else TEST_HOOKS_LIB_PATH if test_hooks else BENCH_LIB_PATH if bench else LIB_PATH
    if not force and not _stale(lib, bench):
        return lib
    build_dir = BUILD_DIR + ("_trace" if trace else "_testhooks" if test_hooks else "_bench" if bench else "")
    os.makedirs(build_dir, exist_ok=True)
    objs = []
    extra = ["-Xptxas", "-v"] if verbose else []
    if trace:
        extra += ["-DGQA_TRACE"]
    if test_hooks:
        extra += ["-DGQA_TEST_HOOKS"]
    procs = []
    for src in sources(bench):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        objs.append(obj)
    failed = False
    for cmd, pr in procs:
        out, _ = pr.communicate()
        if out and (verbose or pr.returncode != 0):
            sys.stdout.write(out)
        if pr.returncode != 0:
            failed = True
            sys.stdout.write("FAILED: " + " ".join(cmd) + "\n")
    if failed:
        raise RuntimeError(f"nvcc failed building {os.path.basename(lib)}")
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcuda"], check=True)
    os.replace(tmp, lib)
    return lib


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--trace", action="store_true")
    ap.add_argument("--test-hooks", action="store_true")
    ap.add_argument("--bench", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, trace=a.trace, test_hooks=a.test_hooks, bench=a.bench))


if __name__ == "__main__":
    main()
