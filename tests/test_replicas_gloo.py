"""bench.py's multi-rank logic on CPU with two gloo ranks (no GPU).

The build does not shard: under torchrun every rank builds its own replica,
the job's time is the slowest rank's, and the value counts every rank's
particles.  The reference arm runs on rank 0 only.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]                      # rank 1 is the slow replica
        worst = bench.max_over_ranks(local_ms, dist)
        bench.barrier(dist)
        buf = io.StringIO()
        with redirect_stdout(buf):                       # the reference arm prints on rank 0 only
            if rank != 0:
                bench.run_reference(type("A", (), {"scene": "tiny", "steps": 1, "warmup": 1, "gpus": world,
                                                   "reference_budget": 5.0, "stable": False})())
        out[rank] = (worst, buf.getvalue())
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time_and_reference_runs_on_rank_zero_only():
    port = _free_port()
    with mp.Manager() as manager:
        out = manager.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][0] == 5.0 and res[1][0] == 5.0
    assert res[1][1] == "", "a non-zero rank of the reference arm prints nothing"


def test_value_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench

    # two replicas of 1M particles whose slowest step takes 50 us: 40,000 Mparticles/s
    assert abs(bench.job_rate(2, 1_000_000, 0.05) - 40_000.0) < 1e-6
    assert abs(bench.job_rate(1, 1_000_000, 0.05) - 20_000.0) < 1e-6
