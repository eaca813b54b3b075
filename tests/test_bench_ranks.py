"""The benchmark's multi-rank path on the CPU: two gloo ranks stand in for two GPUs.

Each rank of bench.py runs the same per-GPU workload (replicas); the slowest rank's time is
taken with an all-reduce MAX and the whole-job throughput counts every rank's work. The
reference arm runs on rank 0 alone; the other ranks exit without printing."""
import multiprocessing
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(1.5 + rank, dist, "cpu")  # rank r "took" 1.5 + r ms
        dist.barrier()
        out.put((rank, slowest, bench.job_throughput(1e12, 10, world, slowest)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    ctx = multiprocessing.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = [out.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    assert [r for r, _, _ in results] == [0, 1]
    for _, slowest, tput in results:
        assert slowest == 2.5  # both ranks see the slowest rank's time
        # 1e12 FLOP per rank and step, 10 steps, 2 ranks, 2.5 ms -> 8000 TFLOP/s
        assert tput == pytest.approx(8000.0)


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25
    assert bench.job_throughput(2e12, 5, 1, 10.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
