"""The bench's own arm on a GPU prints the contract's JSON line: the headline metric on the full-depth eviction, with
roofline, end-to-end and clock objects and the count of the library's launches.  (`--no-extra` skips the extra
workloads and the CPU baseline, which tests/test_bench_contract.py covers through the reference arm.)"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line(gpu):
    r = subprocess.run([sys.executable, "bench.py", "--steps", "4", "--warmup", "3", "--no-extra", "--preroll", "0.2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in line, key
    assert line["unit"] == "GB/s" and line["value"] > 0 and line["n_gpus"] == 1 and line["steps"] == 4
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["vs_baseline"] is None
    assert line["config"]["workload"] == "full_depth_bf16_single_eviction"
    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert rf["traffic"] is None or rf["traffic"] > 0
    e2e = line["e2e"]
    assert e2e["unit"] == "GB/s" and e2e["value"] > 0
    assert e2e["h2d_bytes_per_step"] == 2 * 6240 * 64 * 4 and e2e["d2h_bytes_per_step"] == 4
    assert line["gpu_launches"] == 2 * line["steps"]  # scan + gather per step (the history is empty)
    clk = line["clocks"]
    assert "sm_mhz" in clk and "reasons" in clk
