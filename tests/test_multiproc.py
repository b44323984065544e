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


def test_reference_and_gpu_arms_describe_the_same_workload():
    """bench.py's two arms build their `config` object with one function, so
    the reference line and the GPU line name the same workload."""
    import bench
    import synthetic
    wl = dict(synthetic.WORKLOADS[bench.DEFAULT_WORKLOAD])
    a = bench.bench_config(wl, bench.DEFAULT_WORKLOAD, {}, 1)
    b = bench.bench_config(wl, bench.DEFAULT_WORKLOAD, {}, 1)
    assert a == b and a["workload"].startswith("matmul_reduce_scatter W=4 M=4096 N=4096 K=4096 f16")
    assert {"l2", "parallelism", "op", "M", "N", "K", "seed", "dist"} <= set(a)
    assert bench.bench_config(wl, bench.DEFAULT_WORKLOAD, {}, 2)["parallelism"] == "replicas x2"


def test_recorded_traffic_is_used_only_on_the_kernel_source_it_was_taken_on(tmp_path, monkeypatch):
    """The bench line's roofline.traffic comes from a committed ncu record
    only while the kernel sources hash to the value stored beside it."""
    import bench
    csrc = tmp_path / "gemm_collective_tiles_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cuh").write_text("kernel v1\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = tmp_path / "profiles" / "traffic_w.txt"
    rec.write_text(f"# one launch\ndram_bytes_per_launch: 123456\nkernel_source_sha256_16: {bench.kernel_source_hash()}\n")
    assert bench.recorded_traffic("w") == 123456
    (csrc / "k.cuh").write_text("kernel v2\n")
    assert bench.recorded_traffic("w") is None
    assert bench.recorded_traffic("absent") is None
