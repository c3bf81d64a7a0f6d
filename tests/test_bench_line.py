"""The JSON line bench.py prints: every key the measurement contract asks
for, with values of the right kind, for our arm (on the GPU, the tiny
workload) and for the reference arm (the fp64 oracle on the host cores)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e"]


def _run(args, timeout=900):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def _check_base(d):
    for k in BASE_KEYS:
        assert k in d, k
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["config"]["workload"] == "tiny"
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] >= 0 and e["d2h_bytes_per_step"] >= 0


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "1"])
    _check_base(d)
    assert d["impl"] == "reference" and d["dtype"] == "f64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_our_arm_line():
    d = _run(["--workload", "tiny", "--steps", "5", "--warmup", "3", "--e2e-steps", "3"])
    _check_base(d)
    assert "impl" not in d or d["impl"] != "reference"
    assert d["dtype"] == "f16" and d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["achieved"] > 0 and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    c = d["clocks"]
    for k in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert k in c, k
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
