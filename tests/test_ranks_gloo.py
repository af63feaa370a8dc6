"""The multi-rank side of the benchmark on host processes (gloo, world size 2): the ranks meet
only in barriers and in the max over ranks of the timed region, and the whole-job rate is the
units of every rank over the slowest rank's time. No GPU is used."""

import importlib.util
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _load_bench():
    spec = importlib.util.spec_from_file_location("kda_bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.argv = ["bench.py"]
    bench = _load_bench()
    ranks = bench.Ranks(world, backend="gloo", device="cpu")
    ranks.barrier()
    ms = 10.0 * (rank + 1)                      # rank r "took" 10 (r + 1) ms
    slowest = ranks.max(ms)
    rate = ranks.job_throughput(1000.0, ms)     # 1000 units per rank
    ranks.barrier()
    ranks.close()
    out.put((rank, slowest, rate))


def test_two_gloo_ranks_take_the_max_and_sum_the_units():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, rate in results:
        assert slowest == pytest.approx(20.0)           # max over ranks, seen by every rank
        assert rate == pytest.approx(2 * 1000.0 / 0.020)  # both ranks' units over the slowest time


def test_world_size_must_match_gpus(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "0")
    bench = _load_bench()
    with pytest.raises(SystemExit):
        bench.Ranks(1, backend="gloo", device="cpu")


def test_reference_arm_prints_nothing_on_other_ranks(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    bench = _load_bench()
    bench.run_reference(bench.parse(["--impl", "reference", "--gpus", "2"]))
    assert capsys.readouterr().out == ""
