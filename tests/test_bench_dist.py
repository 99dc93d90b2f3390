"""The benchmark's multi-rank logic on CPU: two gloo ranks, each timing its
own replica; the job takes the slowest rank's time and sums the tokens."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [10.0, 25.0][rank]
        tmax, value = bench.combine_ranks(dist, ms, 8192, "cpu")
        out[rank] = (tmax, value)
        # the reference arm runs on rank 0 only; the others return without work
        class A:
            workload, steps, warmup, ref_budget = "single_token", 1, 0, 0.1
        r = bench.run_reference(A, rank, world)
        out[10 + rank] = r is None
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        tmax, value = res[r]
        assert tmax == 25.0
        assert value == pytest.approx(2 * 8192 / 0.025)
    assert res[10] is False and res[11] is True


def test_single_process():
    import bench
    tmax, value = bench.combine_ranks(None, 4.0, 1000)
    assert tmax == 4.0 and value == pytest.approx(250000.0)
