"""The benchmark's JSON line on a GB300: one line with every key of the
contract, a consistent roofline and an end-to-end figure from host buffers."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_main_line_has_every_contract_key():
    r = subprocess.run([sys.executable, "bench.py", "--main-only", "--no-cpu-baseline",
                        "--steps", "5", "--warmup", "3"], cwd=ROOT, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1, lines
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["value"] > 0
    assert d["config"]["workload"] == "llama3-8b-decode" and "l2" in d["config"]
    roof = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in roof, key
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    e2e = d["e2e"]
    assert e2e["unit"] == d["unit"] and 0 < e2e["value"] <= d["value"] * 1.05
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == d["detail"]["kernels_per_step"] * d["steps"]
    assert d["clocks"]["sm_mhz"] is not None
