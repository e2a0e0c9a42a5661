"""The multi-rank path of bench.py on CPU: two gloo ranks, as torchrun would
start them on two GPUs (each rank its own batch, no collective on the data
path; the barrier and a max over ranks of the timed region are the only
communication)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        # rank r "took" (r + 1) ms per step and 10 (r + 1) ms end to end
        step_ms, e2e_ms = bench.max_over_ranks([rank + 1.0, 10.0 * (rank + 1)], dist, "cpu")
        value = bench.job_tflops(world, 2e12, step_ms)
        q.put((rank, step_ms, e2e_ms, value))
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_time_and_the_whole_job_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, step_ms, e2e_ms, value in got:
        assert step_ms == 2.0 and e2e_ms == 20.0          # both ranks see the slowest rank
        assert value == pytest.approx(2 * 2e12 / 2e-3 / 1e12)  # 2 ranks x their work / slowest time


def test_single_rank_needs_no_group():
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.job_tflops(1, 1e12, 1.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    """Under torchrun the reference arm's other ranks exit without work."""
    from memory_efficient_cnn_gb300 import workloads as wl

    class A:
        steps, warmup = 1, 0

    bench.run_reference(A(), wl.TINY, rank=1, world=2)
    assert capsys.readouterr().out == ""
