"""Host logic of the multi-process bench: independent replicas whose job time
is the slowest rank's, combined over a world-size-2 gloo group on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, value = bench.combine_over_ranks(times[rank], units_per_step=64, steps=100,
                                             world=world, device="cpu")
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_sum_units():
    world, times = 2, [40.0, 50.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, value in got:
        assert ms == pytest.approx(50.0)                        # max over ranks
        assert value == pytest.approx(2 * 64 * 100 / 0.050)     # all ranks' units / job time


def test_single_process_needs_no_group():
    ms, value = bench.combine_over_ranks(25.0, units_per_step=64, steps=10, world=1, device="cpu")
    assert ms == 25.0 and value == pytest.approx(64 * 10 / 0.025)


def test_reference_arm_runs_on_rank_zero_only():
    class A:
        steps, warmup = 1, 0
    assert bench.run_reference(A(), rank=1, world=2) is None
