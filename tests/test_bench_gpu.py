"""bench.py on a GPU: one small run prints a JSON line with every field of its contract."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _line(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_bench_line_carries_the_contract_fields():
    # a small workload larger than L2 (16.8 MB in 24 rotating copies): the tiny one would need thousands
    d = _line("--workload", "t5xxl_sweep_G1", "--secondary", "none", "--steps", "3", "--warmup", "3",
              "--e2e-steps", "2", "--repeat-seconds", "0.05")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == "t5xxl_sweep_G1"
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0 and r["readonly_peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0 and cpu["cores_1"]["cores"] == 1
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 2 * d["steps"] * d["timing"]["blocks"]   # decode + split-combine per step
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]


def test_bench_meanpool_line():
    d = _line("--variant", "meanpool", "--workload", "tiny", "--steps", "3", "--warmup", "3", "--e2e-steps", "2",
              "--repeat-seconds", "0.05", "--no-cpu-baseline")
    assert d["config"]["workload"] == "meanpool_tiny" and d["dtype"] == "f32" and d["value"] > 0
    assert d["roofline"]["kernel"] == "meanpool_kernel"
