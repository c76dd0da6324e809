"""The benchmark's JSON line keeps its contract: one line on stdout with the metric, the
whole-job value and its step time, the roofline of the dominant kernel (achieved / measured
peak), the end-to-end figure with the bytes copied each way, the kernel launch count, the clock
record and the workload's config.  A short run (3 timed steps, no sweep, no CPU baseline)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_json_line_contract():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3",
                        "--no-sweep", "--no-cpu-baseline", "--e2e-steps", "3"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-4000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])

    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches",
              "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["data"].startswith("synthetic") and "workload" in d["config"]
    # value: whole-job tokens/s from the mean step time (4096 tokens a step)
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert abs(d["value"] * d["ms_per_step"] / 1e3 - 4096) / 4096 < 1e-6

    roof = d["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert roof["achieved"] > 0 and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    assert roof["traffic"] is None or roof["traffic"] > 0

    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == "tokens/s"
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["value"] < d["value"]          # the host copies are inside its timed region

    assert d["gpu_launches"] == 3 * d["steps"]   # layout, NVFP4 dispatch, combine per step
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
