"""bench.py prints the one JSON line its consumers parse: the keys and types
are checked here, the reference arm on CPU and the default arm on a GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, timeout=600):
    out = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def _common(d):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["vs_baseline"] is None and d["data"] == "synthetic"
    assert d["warmup"] >= 3
    assert isinstance(d["config"]["workload"], str)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    assert cb["unit"] == d["unit"] and isinstance(cb["sample"], str)


def test_reference_arm_line():
    d = _bench("--impl", "reference", "--workload", "f32_B1_H1_N128_d64", "--steps", "2",
               "--warmup", "3")
    _common(d)
    assert d["impl"] == "reference" and d["dtype"] == "f64"
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


@pytest.mark.gpu
def test_default_arm_line():
    d = _bench("--steps", "3", "--warmup", "3", "--cpu-budget", "1")
    _common(d)
    assert d["config"]["workload"] == "bf16_B1_H32_N16384_d128_causal"
    assert d["n_gpus"] == 1 and d["dtype"] == "bf16" and d["unit"] == "TFLOP/s"
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["peak"] > 0 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert r["traffic"] is None or r["traffic"] > 0
    e = d["e2e"]
    assert e["unit"] == "TFLOP/s" and 0 < e["value"] <= d["value"] * 1.05
    assert e["h2d_bytes_per_step"] == 3 * 32 * 16384 * 128 * 2
    assert e["d2h_bytes_per_step"] == 32 * 16384 * 128 * 2 + 32 * 16384 * 4
    assert d["gpu_launches"] >= d["steps"]
    assert abs(r["frac_of_nominal_dense"] - r["achieved"] / 2250.0) < 1e-9
    c = d["clocks"]
    assert c["sm_max_mhz"] > 0 and isinstance(c["reasons"], list)
    assert c["period_ms"] == 10 and isinstance(c["samples_in_timed_region"], int)
    assert d["memory"]["extra_device_bytes_per_call"] == 0
