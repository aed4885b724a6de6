"""The multi-GPU path of bench.py on CPU: two ranks over gloo.

bench.py runs one replica of the workload per rank (weak scaling, no
collective on the data path), brackets the timed region with barriers and
reports the slowest rank's time; the whole-job throughput counts every rank's
units. The same helpers run here with the gloo backend on CPU tensors."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        slowest = bench.max_over_ranks(times[rank], "cpu")
        dist.barrier()
        out[rank] = (slowest, bench.whole_job_rate(1000.0, dist.get_world_size(), slowest))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(0.25, 0.5), (0.75, 0.125)])
def test_two_ranks_report_the_slowest_rank(times):
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    slowest = max(times)
    for r in range(world):
        assert res[r][0] == slowest
        assert res[r][1] == pytest.approx(1000.0 * world / slowest)


def test_one_rank_needs_no_process_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(0.3, "cpu") == 0.3
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0
