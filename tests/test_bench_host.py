"""Host-side figures that bench.py reports beside the timings (no GPU): the
padded MMA rows the kernels execute and the per-step percentiles."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
from synthetic import WORKLOADS, make_routing  # noqa: E402


def test_padded_slots_equal_the_aligned_length():
    # the rows the GEMMs run are the align step's num_tokens_post_padded
    rng = np.random.default_rng(3)
    wl = WORKLOADS["deepseek_v3"]
    for block in (16, 32, 64, 128):
        for M in (1, 7, 64):
            ids = rng.integers(-2, wl.E + 2, size=(M, wl.topk)).astype(np.int32)  # some out of range
            _, _, npp, _ = oracle.moe_align_block_size(ids.reshape(-1), wl.E, block)
            ex = bench.executed_work(wl, ids, block)
            assert ex["padded_slots"] == int(np.asarray(npp).reshape(-1)[0])
            assert ex["executed_flops"] == 6 * ex["padded_slots"] * wl.H * wl.I


def test_executed_work_on_a_workload_routing():
    wl = WORKLOADS["mixtral8x7b"]
    ids, _ = make_routing(wl, 16, 1016)
    ex = bench.executed_work(wl, np.asarray(ids), 16)
    alg = bench.algorithmic(wl, 16, np.asarray(ids))
    # 32 routed pairs over 8 experts, each padded to 16 rows: at least one block per touched expert
    assert 32 <= ex["padded_slots"] <= 32 + alg["touched"] * 15
    assert ex["padded_slots"] % 16 == 0
    assert ex["executed_flops"] >= alg["layer_flops"]


def test_step_percentiles():
    ms = np.arange(1, 101, dtype=np.float64) / 1000.0  # 1 .. 100 us
    st = bench.step_stats(ms)
    assert st["median"] == 50.5
    assert abs(st["p10"] - 10.9) < 1e-9 and abs(st["p90"] - 90.1) < 1e-9
