"""The multi-rank host logic of bench.py on CPU: two gloo ranks (replicas only,
no collective on the data path; the only collective is the timing maximum)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r was slower on the first timing, faster on the second
        got = bench.max_over_ranks([10.0 + rank, 20.0 - rank], world, "cpu")
        value = bench.whole_job_tflops(2e12, 5, got[0], world)
        out[rank] = (got[0], got[1], value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_work():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        ms0, ms1, value = res[r]
        assert ms0 == 11.0 and ms1 == 20.0          # max over the ranks, on every rank
        assert value == pytest.approx(2 * 2e12 * 5 / 11e-3 / 1e12)


def test_one_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1, "cpu") == [3.0, 4.0]
    assert bench.whole_job_tflops(1e12, 2, 4.0, 1) == pytest.approx(1e12 * 2 / 4e-3 / 1e12)
