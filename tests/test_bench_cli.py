"""bench.py's reference arm (the CPU oracle) on small workloads: one JSON line with the contract's keys."""
import importlib.util
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench_module():
    spec = importlib.util.spec_from_file_location("bench_cli", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=600, check=True)
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    return json.loads(lines[0])


def _check_contract(d, steps, warmup):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == steps and d["warmup"] == warmup
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]


def test_reference_arm_decode_tiny():
    d = _run("--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3")
    _check_contract(d, 3, 3)
    assert d["config"]["workload"] == "tiny" and d["dtype"] == "f64"


@pytest.mark.parametrize("wl,name", [("tiny", "meanpool_tiny"), ("t5xxl_sweep_G4", "meanpool_t5xxl_G4")])
def test_reference_arm_meanpool(wl, name):
    d = _run("--impl", "reference", "--variant", "meanpool", "--workload", wl, "--steps", "3", "--warmup", "3")
    _check_contract(d, 3, 3)
    assert d["config"]["workload"] == name and d["dtype"] == "f32" and d["cpu_baseline"]["cores"] == 1
    H, G, h, dm = (d["config"][k] for k in ("H", "G", "h", "d_model"))
    assert d["config"]["bytes_per_step"] == (H + G) * h * dm * 4


def test_meanpool_workloads():
    b = _bench_module()
    assert b.meanpool_workload("tiny") == ("meanpool_tiny", {"H": 8, "G": 2, "h": 64, "d_model": 512, "config_id": 0})
    name, shp = b.meanpool_workload("t5xxl_sweep_G1")
    assert name == "meanpool_t5xxl_G1" and (shp["H"], shp["G"], shp["h"], shp["d_model"]) == (64, 1, 64, 4096)
    name, shp = b.meanpool_workload("t5xxl_checkpoint")   # the default: 144 projections in one call
    assert name == "meanpool_t5xxl_checkpoint" and shp["outer"] == 144 and (shp["H"], shp["G"]) == (64, 8)
    assert b.MEANPOOL_DEFAULT == "t5xxl_checkpoint"
    with pytest.raises(SystemExit):
        b.meanpool_workload("mistral7b")
