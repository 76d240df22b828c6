"""GPU parity of moe_align_block_size: bit-exact against the oracle."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import weight_quantized_moe_align_gb300 as w
from synthetic import WORKLOADS, make_routing

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "align_cases.json")


@pytest.fixture(scope="module", autouse=True)
def built():
    w.build()
    w.load()


def run_align(ids_np, E, B):
    ids = torch.as_tensor(np.asarray(ids_np, dtype=np.int32), device=DEV)
    assert ids.dim() == 2
    status = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    s, e, npp, cnt = w.moe_align_block_size(ids, E, B, status=status)
    torch.cuda.synchronize()
    return s.cpu().numpy(), e.cpu().numpy(), int(npp.item()), cnt.cpu().numpy(), int(status.item())


def compare(ids, E, B):
    ids = np.asarray(ids, dtype=np.int32)
    if ids.ndim == 1:
        ids = ids.reshape(-1, 1)
    s, e, npp, cnt, st = run_align(ids, E, B)
    rs, re_, rnpp, rcnt = oracle.moe_align_block_size(ids, E, B)
    assert npp == rnpp
    assert np.array_equal(s, rs)
    assert np.array_equal(e, re_)
    assert np.array_equal(cnt, rcnt)
    bad = bool(np.any((ids < 0) | (ids >= E)))
    assert st == (w.DEV_BAD_EXPERT_ID if bad else 0)


def test_golden_cases():
    with open(GOLDEN) as f:
        for c in json.load(f)["cases"]:
            if not c["ids"]:
                continue  # M = 0 is covered by the layer tests
            ids = np.array(c["ids"], dtype=np.int32)
            s, e, npp, cnt, st = run_align(ids, c["E"], c["block"])
            assert s.tolist() == c["sorted_ids"], c["name"]
            assert e.tolist() == c["expert_ids"], c["name"]
            assert npp == c["num_tokens_post_padded"], c["name"]
            assert cnt.tolist() == c["expert_counts"], c["name"]


@pytest.mark.parametrize("seed", range(40))
def test_random(seed):
    rng = np.random.default_rng(1000 + seed)
    E = int(rng.choice([1, 3, 8, 16, 64, 160, 256]))
    M = int(rng.integers(1, 3000))
    k = int(rng.integers(1, min(E, 8) + 1))
    B = int(rng.choice([16, 32, 64, 128, 256]))
    compare(rng.integers(0, E, size=(M, k)), E, B)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_routing_every_block(name):
    wl = WORKLOADS[name]
    for M in wl.m_sweep:
        ids, _ = make_routing(wl, M, 1000 + M)
        for B in (16, 32, 64, 128, 256):
            compare(ids.numpy(), wl.E, B)


def test_special_cases():
    compare(np.zeros((4000, 2)), 8, 16)             # one hot expert, many chunks
    compare(np.array([[255]]), 256, 16)              # single pair, last expert
    compare(np.full((3, 4), 5), 8, 64)               # duplicates inside tokens
    compare(np.array([[1, 300], [-4, 2], [7, 7]]), 8, 16)  # invalid ids dropped + status
    compare(np.arange(256).reshape(32, 8) % 256, 256, 16)  # every expert once
    compare(np.random.default_rng(5).integers(0, 256, size=(8192, 2)), 256, 16)  # 16384 pairs


def test_max_pairs_w8_prefill():
    wl = WORKLOADS["mixtral8x22b_w8"]
    ids, _ = make_routing(wl, 8192, 1000 + 8192)
    compare(ids.numpy(), wl.E, 128)
    compare(ids.numpy(), wl.E, 256)


def test_outputs_stay_in_bounds():
    """Canaries right after every output buffer survive the call."""
    rng = np.random.default_rng(9)
    E, B = 64, 32
    ids = torch.as_tensor(rng.integers(0, E, size=(300, 6)).astype(np.int32), device=DEV)
    cap = w.align_capacity(300 * 6, E, B)
    pad = 64
    canary = -123456789
    s = torch.full((cap + pad,), canary, dtype=torch.int32, device=DEV)
    e = torch.full((cap // B + pad,), canary, dtype=torch.int32, device=DEV)
    n = torch.full((1 + pad,), canary, dtype=torch.int32, device=DEV)
    c = torch.full((E + pad,), canary, dtype=torch.int32, device=DEV)
    w.moe_align_block_size(ids, E, B, out=(s, e, n, c))
    torch.cuda.synchronize()
    assert torch.all(s[cap:] == canary) and torch.all(e[cap // B:] == canary)
    assert torch.all(n[1:] == canary) and torch.all(c[E:] == canary)
    rs, re_, rn, rc = oracle.moe_align_block_size(ids.cpu().numpy(), E, B)
    assert np.array_equal(s[:cap].cpu().numpy(), rs) and int(n[0]) == rn
