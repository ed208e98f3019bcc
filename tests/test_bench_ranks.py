"""The multi-rank host logic of bench.py on CPU: two gloo ranks (one process each)
agree on the job's time (the slowest rank's) and rate (all ranks' units over it), and the
reference arm does its work on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        ms_local = 2.0 + rank                          # rank 1 is the slow one
        ms, value = bench.job_rate(ms_local, 1000.0, ws)
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in got:
        assert ms == 3.0
        assert value == pytest.approx(2 * 1000.0 / 3e-3)


def test_single_rank_needs_no_process_group():
    assert bench.job_rate(4.0, 100.0, 1) == (4.0, 100.0 / 4e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(None, bench.wl.CONFIGS["llama3.1-8b-kv"])   # returns before any work
    assert capsys.readouterr().out == ""
