"""`bench.py --impl reference` (the fp64 oracle timed on host cores) on the CPU: one JSON line
with the same metric, unit and workload as the GPU arm, and the keys the line must carry; under
a multi-rank launch only rank 0 prints."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(**env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)


def _json_lines(out):
    return [json.loads(line) for line in out.splitlines() if line.startswith("{")]


def test_reference_arm_prints_one_contract_line():
    r = _run(RANK="0")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1, r.stdout
    d = lines[0]
    sys.path.insert(0, ROOT)
    import bench
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["ms_per_step"] > 0
    assert d["config"]["workload"].startswith("KDA chunked prefill B=4 T=8192 H=32 dk=dv=128")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    r = _run(RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    assert r.returncode == 0, r.stderr[-2000:]
    assert _json_lines(r.stdout) == []


def test_bench_defaults_and_warmup_floor():
    """No flags: one GPU, the headline arm, a bounded number of steps; never fewer than 3
    warm-up steps (a smaller request runs 3 and the line reports 3)."""
    sys.path.insert(0, ROOT)
    import bench
    a = bench.parse([])
    assert a.gpus == 1 and a.impl == "ours" and a.warmup >= 3 and 1 <= a.steps <= 1000 and a.workload is None
    assert bench.parse(["--warmup", "1"]).warmup == 3
    assert bench.parse(["--impl", "reference", "--gpus", "4", "--steps", "7", "--warmup", "9"]).warmup == 9
    with pytest.raises(SystemExit):
        bench.parse(["--steps", "0"])
