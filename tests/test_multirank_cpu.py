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


def test_reference_arm_prints_one_complete_line():
    """bench.py --impl reference on the CPU (one step, no warm-up): one JSON line with the
    contract's keys, the same metric, unit and config as the measured arm."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {kk: vv for kk, vv in os.environ.items() if kk not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], capture_output=True, text=True, timeout=600, env=env, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True and d["value"] > 0 and d["steps"] == 1
    from rational_softmax_attention_gb300.inputs import ATTN_LONG_WIDE, RA_SOFTMAX_LONG_ROWS
    assert d["config"] == json.loads(json.dumps(bench.step_config(ATTN_LONG_WIDE, RA_SOFTMAX_LONG_ROWS)))
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
