"""bench.py's JSON contract, checked on the CPU through the reference arm
(the fp64 oracle on a small row sample of the same workload): one JSON line
with the metric, value, unit, step counts, the cpu_baseline and e2e objects.
The GPU arm prints the same keys plus the kernel measurements; it runs on
the GPU only.
"""

import json
import os
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.timeout(300)
def test_reference_arm_prints_one_contract_line():
    t0 = time.perf_counter()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3", "--ref-rows", "256"],
                       capture_output=True, text=True, cwd=ROOT, timeout=280)
    wall = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["unit"] == "ms" and d["value"] > 0 and d["higher_is_better"] is False
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] and d["config"]["M"] == 220000
    # ms_per_step is what one step actually took: the steps fit in the run's wall time, and value is
    # that time scaled from the sampled rows to all M rows
    rows = d["config"]["sample_rows"]
    assert 0 < rows <= 256
    assert d["steps"] * d["ms_per_step"] * 1e-3 < wall
    assert abs(d["value"] - d["ms_per_step"] * 220000 / rows) <= 1e-3 * d["value"] + 0.1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == "ms"
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
