"""The JSON line of `bench.py --impl reference` (the oracle timed on the host)
carries the keys the bench contract names, on the workload the GPU arm uses."""
from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["config"]["workload"] == "b256"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_cpu_baseline_single_and_all_cores():
    sys.path.insert(0, ROOT)
    import bench
    from device_token_sampling_gb300 import workloads as W
    d = bench.cpu_baseline(W.tiny(), budget_rows=4)
    assert d["kind"] == "oracle" and d["cores"] == 1 and d["value"] > 0
    assert d["all_cores"]["cores"] == (os.cpu_count() or 1) and d["all_cores"]["value"] > 0
