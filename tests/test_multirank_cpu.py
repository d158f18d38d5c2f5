"""The multi-rank parts of bench.py on CPU: world-size-2 `gloo` ranks (spawned
processes, rendezvous on 127.0.0.1) check the max-over-ranks timing and the whole-job
value, and the reference arm's rank 1 exits without work."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, times, out_q):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        step = bench.max_over_ranks(torch, times[rank], world, torch.device("cpu"))
        dist.barrier()
        out_q.put((rank, step, bench.whole_job_rate(world, 1e9, step)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_the_slowest_and_sum_the_work():
    world, times = 2, [31.5, 47.25]  # ms per step on each rank
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, step, rate in res:
        assert step == max(times)  # every rank reports the slowest rank's time
        assert rate == pytest.approx(world * 1e9 / (max(times) / 1e3) / 1e9)


def test_one_rank_is_the_identity():
    assert bench.max_over_ranks(torch, 12.5, 1, None) == 12.5
    assert bench.whole_job_rate(1, 2e9, 10.0) == pytest.approx(200.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = bench.parse_args(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"])
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""
