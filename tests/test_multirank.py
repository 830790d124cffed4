"""The benchmark's multi-rank path on CPU with two gloo ranks: barrier,
max-over-ranks timing and the whole-job aggregate (replicas only: ranks run
independent GEMMs and exchange nothing but the timing)."""

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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench._barrier(world)
    local_ms = 10.0 * (rank + 1)             # rank 1 is the slower one
    mx = bench._barrier_max(local_ms, world)
    q.put((rank, mx, bench.aggregate_tflops(2e12, 4, mx, world)))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, mx, agg in got:
        assert mx == 20.0                     # both ranks see the slowest rank's time
        assert agg == pytest.approx(2 * 2e12 * 4 / 20e-3 / 1e12)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_aggregate_is_whole_job():
    import bench
    # one rank, 137.4 GFLOP per step, 10 steps in 1 ms -> 1374 TFLOPS
    assert bench.aggregate_tflops(137.4e9, 10, 1.0, 1) == pytest.approx(1374.0)
    assert bench.aggregate_tflops(137.4e9, 10, 1.0, 4) == pytest.approx(4 * 1374.0)
