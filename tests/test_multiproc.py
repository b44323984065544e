"""The multi-rank host logic of the benchmark (one independent replica per
GPU): max over ranks of the timed region, whole-job throughput, rank
environment.  World size 2 over gloo on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        env = bench.dist_env()
        m = bench.max_over_ranks(10.0 + rank, dist)
        v = bench.job_throughput(5.5e11, world, 100, m)
        q.put((rank, env, m, v))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, m, v in res:
        assert env == (2, rank, rank)
        assert m == 11.0                                    # the slowest rank's time
        assert v == pytest.approx(5.5e11 * 100 * 2 / 11e-3 / 1e12)


def test_single_process_identity():
    import bench
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.job_throughput(1e12, 1, 10, 10.0) == pytest.approx(1000.0)
