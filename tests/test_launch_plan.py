"""CPU replay of the fused call's launch plan (``wna16_check_launch_plan``).

The library builds the plan of a call (block size, K splits, workspace layout,
tensor maps, grids) without any CUDA call, and replays every role of every CTA
of both GEMM launches, the gather and the combine through the kernels' own
index expressions. Here it runs on the oracle's align output for the routing of
each workload's batches, at the automatic block and at every forced block
size, on a 152-SM device; every TMA box must lie inside its tensor map, every
workspace write inside its region, every routed pair's fp32 rows written once.

The DeepSeek-V3-shaped layer at M = 256 with forced blocks is where launch
failures were recorded on the GPU (with 128-token blocks; those, and 256, are
now refused on layers of more than 16 experts); its plans are checked here.

Planted mistakes (in the align output handed to the checker, never in the
library) must be reported.
"""
import numpy as np
import pytest

import oracle
import weight_quantized_moe_align_gb300 as w
from synthetic import WORKLOADS
from synthetic.workloads import _seed, make_routing

SMS = 152


@pytest.fixture(scope="module", autouse=True)
def built():
    w.build()
    w.load()


def _ids(wl, M):
    ids, _ = make_routing(wl, M, _seed(wl.name, "route", 1000 + M))
    return ids.numpy().astype(np.int32)


def _check(wl, M, block, ids=None, split_k=0, mutate=None):
    ids = _ids(wl, M) if ids is None else ids
    B = block or w.choose_block(M, wl.topk, wl.E)
    srt, exp, npp, _ = oracle.moe_align_block_size(ids, wl.E, B)
    srt, exp = np.array(srt, dtype=np.int32), np.array(exp, dtype=np.int32)
    if mutate is not None:
        srt, exp, npp = mutate(srt, exp, npp)
    return w.check_launch_plan(M, wl.H, wl.I, wl.E, wl.topk, wl.bits, wl.group_size, wl.has_zeros, wl.act_dtype,
                               wl.scale_dtype, ids, srt, exp, npp, block=block, split_k=split_k, sms=SMS)


@pytest.mark.parametrize("block", [0, 16, 32, 64])
def test_deepseek_v3_m256_forced_blocks(block):
    n, report = _check(WORKLOADS["deepseek_v3"], 256, block)
    assert n == 0, report


@pytest.mark.parametrize("name,M,block", [("deepseek_v3", 256, 128), ("deepseek_v3", 1024, 256),
                                          ("qwen2_57b", 128, 128), ("qwen2_57b", 512, 256)])
def test_large_tiles_refused_on_many_expert_layers(name, M, block):
    # 128/256-token tiles on layers with more than 16 experts are refused, as
    # the fused call refuses them (unsupported)
    n, _ = _check(WORKLOADS[name], M, block)
    assert n == -2


CASES = [(name, M) for name in ("mixtral8x7b", "qwen2_57b", "deepseek_v3") for M in WORKLOADS[name].m_sweep]


@pytest.mark.parametrize("name,M", CASES)
def test_sweep_points_automatic_block(name, M):
    n, report = _check(WORKLOADS[name], M, 0)
    assert n == 0, report


@pytest.mark.parametrize("name,M,block", [
    ("mixtral8x7b", 64, 16), ("mixtral8x7b", 256, 128), ("mixtral8x7b", 1024, 256), ("mixtral8x7b", 16, 32),
    ("qwen2_57b", 128, 64), ("qwen2_57b", 512, 64), ("qwen2_57b", 32, 32),
    ("deepseek_v3", 1024, 16), ("deepseek_v3", 1024, 32), ("deepseek_v3", 1024, 64), ("deepseek_v3", 64, 64),
    ("deepseek_v3", 16, 32), ("tiny", 4, 16), ("tiny", 4, 256),
])
def test_forced_blocks(name, M, block):
    n, report = _check(WORKLOADS[name], M, block)
    assert n == 0, report


@pytest.mark.parametrize("split_k", [2, 3, 8])
def test_forced_down_splits(split_k):
    n, report = _check(WORKLOADS["mixtral8x7b"], 16, 0, split_k=split_k)
    assert n == 0, report


def test_int8_large_prefill_plan():
    wl = WORKLOADS["mixtral8x22b_w8"]
    n, report = _check(wl, 1024, 128)
    assert n == 0, report


def test_dropped_ids_plan():
    wl = WORKLOADS["deepseek_v3"]
    ids = _ids(wl, 64)
    ids[3, 2] = -1
    ids[7, 0] = wl.E
    n, report = _check(wl, 64, 32, ids=ids)
    assert n == 0, report


# ---------------------------------------------------------------- planted mistakes

def _dup_pair(srt, exp, npp):
    srt = srt.copy()
    srt[1] = srt[0]
    return srt, exp, npp


def _bad_expert(srt, exp, npp):
    exp = exp.copy()
    exp[0] = 10_000
    return srt, exp, npp


def _short_total(srt, exp, npp):
    return srt, exp, npp - 16


def _wrong_block_expert(srt, exp, npp):
    exp = exp.copy()
    nb = npp // 16
    exp[nb - 1] = (exp[nb - 1] + 1) % 256
    return srt, exp, npp


@pytest.mark.parametrize("mutate", [_dup_pair, _bad_expert, _short_total, _wrong_block_expert])
def test_planted_align_mistakes_are_reported(mutate):
    n, report = _check(WORKLOADS["deepseek_v3"], 16, 16, mutate=mutate)
    assert n > 0
    assert report


def test_rejected_arguments():
    wl = WORKLOADS["tiny"]
    ids = _ids(wl, 4)
    n, _ = w.check_launch_plan(4, wl.H, wl.I, wl.E, wl.topk, 4, 96, 1, "f16", "f16", ids, np.zeros(64, np.int32),
                               np.zeros(4, np.int32), 0, block=16, sms=SMS)
    assert n == -2  # group size 96: unsupported, as the fused call answers
