"""The N > 1 path of bench.py on the CPU: two `gloo` ranks (the shards are
independent (batch, head) problems, so the only collective is the timing
reduction), and the reference arm, which rank 0 alone runs."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench as b

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        job_ms = b.max_over_ranks(times[rank], world)
        out[rank] = (job_ms, b.job_value(1000, 10, world, job_ms))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    times = [3.0, 5.0]
    mp.start_processes(_rank_main, args=(2, _free_port(), times, out), nprocs=2, join=True,
                       start_method="spawn")
    for rank in range(2):
        job_ms, value = out[rank]
        assert job_ms == 5.0  # every rank reports the job's (slowest rank's) time
        assert value == pytest.approx(2 * 1000 * 10 / 5e-3)  # both ranks' units over that time


def test_one_rank_needs_no_process_group():
    assert bench.max_over_ranks(4.5, 1) == 4.5
    assert bench.job_value(100, 2, 1, 1.0) == pytest.approx(2e5)


@pytest.mark.timeout(120)
def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.main(["--impl", "reference", "--workload", "causal", "--gpus", "2", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out.strip() == ""  # the other ranks exit without work or output
