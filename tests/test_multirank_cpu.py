"""The multi-rank path of bench.py without a GPU: world-size-2 gloo ranks on the CPU.

Under torchrun every rank runs the whole step on its own GPU (heads are independent, so the
path has no data exchange); the ranks meet only to time the step.  These tests check that
host logic: the slowest rank's time is every rank's time, the reported value counts the
work of all ranks, each rank reads its place from the launcher's environment, and the
reference arm runs (and prints) on rank 0 only."""
import os
import socket
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(times[rank], dist, torch.device("cpu"))
        value = bench.whole_job_tflops(world, 1e12, 2, slowest)
        out_q.put((rank, slowest, value, bench.dist_env()))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time_and_the_value_counts_every_rank():
    world, port, times = 2, _free_port(), [3.0, 5.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(r[0] for r in results) == [0, 1]
    for rank, slowest, value, env in results:
        assert slowest == 5.0
        # 2 ranks x 2 steps x 1e12 FLOP in 5 ms
        assert value == pytest.approx(2 * 2 * 1e12 / 5e-3 / 1e12)
        assert env == (world, rank, rank)


def test_single_process_keeps_its_own_time():
    assert bench.max_over_ranks(4.25, None, torch.device("cpu")) == 4.25
    assert bench.whole_job_tflops(1, 1e12, 4, 2.0) == pytest.approx(2000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    bench.run_reference(types.SimpleNamespace(steps=1, warmup=0))
    assert capsys.readouterr().out == ""
