"""bench.py's multi-rank host logic on CPU with the gloo backend (world size 2): the
timing reduction takes the slowest rank, the whole-job value counts every rank's units,
and the reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [120.0, 135.5][rank]
        results[rank] = bench.max_over_ranks(local_ms, world, "cpu")
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world, port = 2, _free_port()
    results = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
    assert results[0] == results[1] == 135.5


def test_whole_job_throughput_counts_all_ranks():
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 131072 tokens x 10 steps in 1000 ms (slowest rank) -> 2.62M tokens/s
    assert bench.whole_job_throughput(131072, 10, 2, 1000.0) == pytest.approx(2 * 1310720)
    assert bench.whole_job_throughput(131072, 10, 1, 500.0) == pytest.approx(2621440)


def test_reference_arm_non_zero_rank_exits_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
