"""bench.py prints one JSON line with the keys its readers rely on: the CPU
reference arm here, the GPU arm on a short run of the small workload."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
             "vs_baseline", "dtype", "data", "config", "impl", "e2e"}


def _run(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run("--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "3")
    assert BASE_KEYS <= set(d)
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and "2 steps" in cb["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"].startswith("zero2_psi1000003_nd4")


@pytest.mark.gpu
def test_gpu_arm_line():
    d = _run("--config", "1", "--steps", "5", "--warmup", "3", "--no-cpu-baseline")
    assert BASE_KEYS <= set(d) and {"roofline", "clocks", "gpu_launches"} <= set(d)
    assert d["impl"] == "gb300" and d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["gpu_launches"] >= 5        # one fused launch per step at least
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert abs(d["step_frac_of_nominal"] - d["step_gbs"] / 8000.0) < 1e-3
    assert d["config"]["l2"] == "flushed between steps"
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == 4 * 2 * 1_000_008 and e["d2h_bytes_per_step"] == 2 * 1_000_003
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
