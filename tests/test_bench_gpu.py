"""`bench.py` on a GPU: the default arm prints one JSON line with the keys its contract names
(metric, value, roofline with the measured peak, e2e with the copied bytes, clocks, launch count),
and its numbers are consistent with each other. Short run: a few steps, no sub-workloads."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_default_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--steps", "5", "--warmup", "3", "--decode-steps", "20",
                        "--e2e-steps", "3", "--no-workloads", "--no-cpu-baseline"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = lines[0]
    sys.path.insert(0, ROOT)
    import bench
    assert d["metric"] == bench.METRIC and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["dtype"] == "bf16"
    assert d["data"] == "synthetic" and d["scaling"] == "weak"
    assert d["config"]["workload"].startswith("KDA chunked prefill B=4 T=8192 H=32 dk=dv=128")
    # tokens/s and ms/step describe the same steps: 4 x 8192 tokens per step
    assert d["value"] == pytest.approx(4 * 8192 / (d["ms_per_step"] * 1e-3), rel=1e-6)
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], rel=1e-9)
    assert rf["achieved"] == pytest.approx(rf["alg_bytes_per_launch"] / (rf["kernel_ms"] * 1e-3) / 1e9, rel=1e-6)
    assert 0.05 < rf["frac"] < 1.2  # a plain copy's rate bounds an HBM-bound kernel
    e2e = d["e2e"]
    assert e2e["unit"] == d["unit"] and 0 < e2e["value"] < d["value"]
    assert e2e["h2d_bytes_per_step"] > 1e9 and e2e["d2h_bytes_per_step"] > 2e8
    assert d["gpu_launches"] == d["steps"]
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    dec = d["decode"]
    assert dec["unit"] == "tokens/s" and dec["value"] > 0 and dec["roofline"]["bound"] == "hbm"
