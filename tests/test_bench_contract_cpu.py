"""The JSON line of `bench.py --impl reference` (the fp64 oracle timed on the
host cores, the comparison arm of the benchmark) on CPU: one line, the
contract's keys, the oracle's own rate in `value`, `cpu_baseline` and `e2e`."""
import json
import os
import subprocess
import sys

import bench
from paged_kv_cache_132_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    proc = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"],
                          cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stderr[-2000:]
    lines = [ln for ln in proc.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, proc.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 1
    assert d["higher_is_better"] is True and d["data"] == "synthetic"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert "workload" in d["config"]
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == d["value"] and cpu["unit"] == d["unit"]
    assert cpu["cores"] >= 1 and cpu["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert cpu["cpu_model"] and cpu["nproc"] >= 1
    # the same config object as the repo's own arm prints for this workload
    w = workloads.make("llama8b", device="cpu")
    ours = bench.decode_config(bench.parse_args([]), w, 1, bench.partition_for(bench.parse_args([]), w), 0)
    assert d["config"] == json.loads(json.dumps(ours))
