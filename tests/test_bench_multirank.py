"""Host logic of the multi-GPU benchmark on CPU: two gloo ranks.

Every rank runs its own replica (no collective on the data path); the only exchange
is the max-over-ranks of the step time that the whole-job throughput divides by.
"""

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 2.0 + 1.5 * rank              # rank 1 is the slow one
        ms_max = bench.world_max(ms, torch.device("cpu"))
        value = bench.aggregate_value(3.0e11, world, ms_max)
        queue.put((rank, ms_max, value))
    finally:
        torch.distributed.destroy_process_group()


def test_single_process_needs_no_group():
    assert bench.world_max(1.25, torch.device("cpu")) == 1.25
    # 2e11 units in 2 ms on one rank -> 100 T units/s
    assert bench.aggregate_value(2.0e11, 1, 2.0) == pytest.approx(100.0)


def test_two_gloo_ranks_take_the_slowest_step():
    world = 2
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, queue)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, value in results:
        assert ms_max == pytest.approx(3.5)            # every rank sees the slowest rank
        # whole-job: both ranks' units over the slowest step (weak scaling)
        assert value == pytest.approx(2 * 3.0e11 / 3.5e-3 / 1e12)
