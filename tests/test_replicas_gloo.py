"""The multi-GPU path of bench.py is replicas only (the forward has no
exchange step).  Its host logic (max-reduced timing, whole-job throughput,
barrier) is checked here with two gloo ranks on the CPU."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = [1.5, 2.5][rank]  # rank 1 is the slow one
    bench.barrier(world)
    slowest = bench.max_over_ranks(world, ms)
    results[rank] = (slowest, bench.job_tflops(world, 1e12, slowest))
    dist.destroy_process_group()


def test_two_replicas():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        slowest, value = results[r]
        assert slowest == 2.5
        assert value == pytest.approx(2 * 1e12 / 2.5e-3 / 1e12)


def test_single_process_is_identity():
    import bench

    assert bench.max_over_ranks(1, 3.0) == 3.0
    assert bench.job_tflops(1, 2e12, 1000.0) == pytest.approx(2.0)
