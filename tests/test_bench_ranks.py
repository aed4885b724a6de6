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


def test_gpus_flag_starts_one_rank_per_replica():
    """`bench.py --gpus 2` starts two ranks itself (torch.distributed.run), each
    with its own RANK; rank 0 prints one line for the whole job, timed by the
    slowest rank (--dry-run: CPU tasks over gloo instead of GPU replicas)."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--dry-run", "--steps", "5",
                        "--warmup", "3"], capture_output=True, text=True, timeout=300, env=env, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2
    assert sorted(line["ranks"]) == [0, 1]
    per_rank = line["rank_ms_per_step"]
    assert len(per_rank) == 2 and per_rank[1] > per_rank[0]  # rank r sleeps (r + 1) ms a step
    assert line["ms_per_step"] == pytest.approx(max(per_rank))
    assert line["value"] == pytest.approx(1000.0 * 2 / (line["ms_per_step"] / 1e3))
    assert line["scaling"] == "weak"
