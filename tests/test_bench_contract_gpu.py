"""The JSON line of `bench.py` (the library's arm) on a GPU, a short run:
one line with the contract's keys -- whole-job value, roofline of the decode
call against the measured HBM peak, the oracle's CPU baseline, the end-to-end
leg through host buffers, the kernel launch count and the SM clocks -- and
the same for the prefill workload's line."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks")


def run(*args):
    proc = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert proc.returncode == 0, proc.stderr[-3000:]
    lines = [ln for ln in proc.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, proc.stdout
    return json.loads(lines[0])


def check_common(d, bound, unit):
    for key in KEYS:
        assert key in d, key
    assert d["n_gpus"] == 1 and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["gpu_launches"] > 0
    r = d["roofline"]
    assert r["bound"] == bound and r["unit"] == unit and r["peak"] > 0
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    assert 0.0 < r["frac"] < 1.5
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] > 0 and cpu["cores"] >= 1 and cpu["sample"]
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["clocks"]["sm_max_mhz"] > 0


def test_decode_line():
    d = run("--steps", "20", "--warmup", "3", "--cpu-seconds", "1", "--no-rows")
    check_common(d, "hbm", "GB/s")
    assert d["unit"] == "GB/s" and d["dtype"] == "bf16"
    assert d["decode_gbs"] == pytest.approx(d["roofline"]["achieved"], rel=1e-6)
    assert d["cpu_baseline"]["cpu_model"]
    rows = d["rows"]
    assert rows["host_us_per_decode_call_c_abi"] > 0 and rows["host_us_per_decode_call_python"] > 0
    assert rows["a2_a6_decode_warm_graph_us"] > 0


def test_prefill_line():
    d = run("--workload", "prefill_llama8b", "--steps", "3", "--warmup", "3", "--cpu-seconds", "1")
    check_common(d, "tensor", "TFLOP/s")
    assert d["unit"] == "TFLOP/s" and d["dtype"] == "bf16"
