"""The bench's multi-GPU path on the CPU: replicas only, no collective on the data path.

Under torchrun every rank times its own replica of the workload; the ranks meet at barriers around the timed region,
take the slowest rank's time (a MAX all-reduce) and rank 0 alone prints the line, whose value counts the units of
every rank.  Checked here with two gloo ranks on 127.0.0.1: both ranks see the same slowest time, the whole-job
rate is the world's units over that time, and the reference arm does no work on ranks other than 0.
"""
import argparse
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

# one rank: join the group the way the bench does, then report the slowest time and the whole-job rate
RANK_MAIN = r"""
import json, os, sys
sys.path.insert(0, sys.argv[1])
import bench
dist, rank, world, local = bench._dist()
assert (rank, world, local) == (int(os.environ["RANK"]), 2, int(os.environ["LOCAL_RANK"]))
dist.barrier()
own_ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
slowest = bench._max_over_ranks(dist, own_ms, "cpu")
dist.barrier()
print(json.dumps({"rank": rank, "own": own_ms, "slowest": slowest,
                  "rate": bench.whole_job_rate(world, 400, slowest)}))
dist.destroy_process_group()
"""


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_slowest_time():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), CSA_BENCH_GLOO="1")
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_MAIN, ROOT], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    try:
        for p in procs:
            outs.append(p.communicate(timeout=180))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    for p, (out, errs) in zip(procs, outs):
        assert p.returncode == 0, errs[-2000:]
    res = sorted((json.loads(out.strip().splitlines()[-1]) for out, _ in outs), key=lambda r: r["rank"])
    assert [r["own"] for r in res] == [10.0, 15.0]
    assert all(r["slowest"] == 15.0 for r in res)  # every rank reports the slowest rank's time
    # weak scaling: 2 ranks x 400 units in 15 ms
    assert res[0]["rate"] == pytest.approx(2 * 400 / 0.015)


def test_whole_job_rate_counts_every_rank():
    assert bench.whole_job_rate(1, 400, 1000.0) == pytest.approx(400.0)
    assert bench.whole_job_rate(8, 400, 1000.0) == pytest.approx(3200.0)
    # the same per-rank work at twice the slowest time halves the rate
    assert bench.whole_job_rate(4, 400, 2000.0) == pytest.approx(800.0)


def test_single_process_needs_no_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    dist, rank, world, local = bench._dist()
    assert (dist, rank, world, local) == (None, 0, 1, 0)
    assert bench._max_over_ranks(None, 12.5, "cpu") == 12.5


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(bench, "run_oracle_processes",
                        lambda *a, **k: pytest.fail("rank 1 started the oracle"))
    assert bench.run_reference(argparse.Namespace(warmup=3, steps=5)) is None
    assert capsys.readouterr().out == ""
