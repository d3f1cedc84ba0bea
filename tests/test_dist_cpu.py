"""Multi-rank host logic of bench.py on CPU with the gloo backend (world size 2).

Attention shards into independent (batch, head) work with no exchange step, so bench.py runs
the same per-GPU workload on every rank (weak scaling, no data-path collective). What is
collective is the timing: a barrier and the maximum time over ranks. These tests run that
logic on two CPU processes.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    try:
        dist.barrier()
        got = bench.rank_max(10.0 * (rank + 1) + 0.5, dist, "cpu")
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_rank_max_takes_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = dict(q.get(timeout=5) for _ in range(world))
    assert results == {0: 20.5, 1: 20.5}


def test_rank_max_without_process_group_is_identity():
    import bench

    assert bench.rank_max(3.25) == 3.25


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 3, 3

    bench.run_reference(Args())  # returns at once: no work, no output on ranks other than 0
    assert capsys.readouterr().out == ""


def test_small_config_oracle_timings(monkeypatch):
    # The cpu_baseline leg times the oracle on the small configurations with all cores and, in
    # a child process with the BLAS thread variables set to 1, with one thread.
    import subprocess
    import json

    import bench

    monkeypatch.setattr(bench, "SMALL_CONFIGS", bench.SMALL_CONFIGS[:1])
    rows = bench._time_small_configs(repeats=1)
    assert [r["config"] for r in rows] == ["B=1 H=1 N=256 d=64 non-causal fwd"] and rows[0]["seconds"] > 0

    seen = {}

    def fake_run(cmd, env, **kw):
        seen["cmd"], seen["env"] = cmd, env
        return subprocess.CompletedProcess(cmd, 0, stdout=json.dumps([{"config": "x", "seconds": 0.5}]) + "\n")

    monkeypatch.setattr(bench.subprocess, "run", fake_run)
    out = bench.small_config_timings()
    assert seen["cmd"][-1] == "--small-configs-child"
    assert all(seen["env"][v] == "1" for v in bench.THREAD_VARS)
    assert out["rows"][0]["seconds_1_thread"] == 0.5 and out["rows"][0]["seconds_all_cores"] > 0
