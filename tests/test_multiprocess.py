"""The multi-rank path of bench.py on CPU: world size 2 over gloo (replicas, no
collective on the data path; only the timing is reduced across ranks)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) * 100 ms for 10 steps of 16 tokens
        total, value = bench.aggregate_ranks((rank + 1) * 100.0, 16, 10, dist)
        results[rank] = (total, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_rank_and_value_counts_all_ranks():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        res = dict(results)
    for rank in range(world):
        total, value = res[rank]
        assert total == 200.0  # the slower rank
        assert value == pytest.approx(world * 16 * 10 / 0.2)


def test_single_process_aggregate_is_the_local_figure():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.aggregate_ranks(50.0, 8, 5) == (50.0, 8 * 5 / 0.05)


def test_reference_arm_prints_on_rank_zero_only():
    # the oracle arm on a rank other than 0 does no work and prints nothing
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--M", "4", "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--M", "4", "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-500:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
