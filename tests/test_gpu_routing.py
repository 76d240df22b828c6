"""GPU parity of wna16_topk_routing against the oracle.

Ids are compared exactly: the kernel ranks experts on the exact input logits,
as the oracle does. The one floating-point decision is the group score (sum
of two scores, fp32 on the GPU, fp64 in the oracle): rows whose kept/dropped
group boundary lies within 1e-5 of a tie are checked for validity instead
(every kept group within the tolerance of the boundary, the experts the top-k
of the kept groups). Weights: fp32 against fp64, rtol 1e-5.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import weight_quantized_moe_align_gb300 as w
from synthetic import WORKLOADS, make_router_logits, routing_params

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL_GROUP = 1e-5
_TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def built():
    w.build()
    w.load()


def _as_dtype(logits64, dt):
    """Logits rounded to dtype; returns (device tensor, exact float64 values)."""
    t = torch.as_tensor(np.asarray(logits64, dtype=np.float32)).to(_TORCH[dt])
    return t.to(DEV), t.double().numpy()


def _check(logits64, topk, scoring, renorm, n_groups=1, topk_groups=1, dt="f32", max_ambiguous=0.01):
    x, exact = _as_dtype(logits64, dt)
    ids, wt = w.topk_routing(x, topk, scoring, renorm, n_groups, topk_groups)
    torch.cuda.synchronize()
    ids, wt = ids.cpu().numpy(), wt.cpu().numpy().astype(np.float64)
    rids, rw = oracle.topk_routing(exact, topk, scoring, renorm, n_groups, topk_groups)
    M, E = exact.shape
    ambiguous = np.zeros(M, dtype=bool)
    if n_groups > 1 and topk_groups < n_groups:
        gsc = oracle.routing_group_scores(exact, scoring, n_groups)
        gsc = np.where(np.isnan(gsc), -np.inf, gsc)
        srt = -np.sort(-gsc, axis=1)
        gap = srt[:, topk_groups - 1] - srt[:, topk_groups]
        ambiguous = ~(gap > TOL_GROUP * np.maximum(1.0, np.abs(srt[:, topk_groups - 1])))
    ok = ~ambiguous
    assert np.array_equal(ids[ok], rids[ok])
    np.testing.assert_allclose(wt[ok], rw[ok], rtol=1e-5, atol=1e-6, equal_nan=True)
    assert ambiguous.sum() <= max(1, max_ambiguous * M)
    if ambiguous.any():
        gs = E // n_groups
        sc = oracle.routing_scores(exact, scoring)
        for t in np.nonzero(ambiguous)[0]:
            _check_valid_grouped_row(exact[t], sc[t], gsc[t], ids[t].tolist(), wt[t], topk, renorm, topk_groups, gs)
    return ids, wt


def _ranked(logits_row, allowed):
    key = lambda e: (math.inf if math.isnan(logits_row[e]) else -logits_row[e], e)
    return sorted(allowed, key=key)


def _check_valid_grouped_row(l, sc, gsc, row, wt, topk, renorm, topk_groups, gs):
    """A near-tied group boundary: the GPU's ids must be the top-k of some set of
    topk_groups groups, each within the tolerance of the boundary score."""
    n_groups = len(gsc)
    assert len(set(row)) == topk and all(0 <= e < n_groups * gs for e in row)
    boundary = -np.sort(-gsc)[topk_groups - 1]
    eligible = [g for g in range(n_groups) if gsc[g] >= boundary - 2 * TOL_GROUP * max(1.0, abs(boundary))]
    used = sorted({e // gs for e in row})
    assert len(used) <= topk_groups and all(g in eligible for g in used)
    # pad with the eligible groups whose best expert ranks lowest: if any padding
    # makes the selection the top-k of the kept groups, this one does
    order = {e: i for i, e in enumerate(_ranked(l, range(n_groups * gs)))}
    extra = sorted((g for g in eligible if g not in used),
                   key=lambda g: -min(order[e] for e in range(g * gs, (g + 1) * gs)))
    kept = used + extra[:topk_groups - len(used)]
    allowed = [e for g in kept for e in range(g * gs, (g + 1) * gs)]
    assert _ranked(l, allowed)[:topk] == row
    ew = sc[row] / sc[row].sum() if renorm else sc[row]
    np.testing.assert_allclose(wt, ew, rtol=1e-5, atol=1e-6)


CONFIGS = [
    # E, topk, scoring, renorm, n_groups, topk_groups
    (8, 2, "softmax", True, 1, 1),       # Mixtral
    (64, 8, "softmax", False, 1, 1),     # Qwen2-57B
    (256, 8, "sigmoid", True, 8, 4),     # DeepSeek-V3
    (256, 8, "softmax", True, 8, 3),
    (160, 6, "softmax", False, 8, 3),    # 5 experts per lane
    (40, 4, "sigmoid", False, 1, 1),
    (100, 3, "sigmoid", True, 4, 2),
    (6, 2, "sigmoid", True, 3, 1),
    (256, 32, "softmax", True, 1, 1),    # largest topk
    (256, 8, "sigmoid", True, 32, 4),    # 32 groups of 8
    (1, 1, "softmax", True, 1, 1),
    (32, 32, "sigmoid", False, 1, 1),    # topk = E
    (256, 8, "sigmoid", True, 4, 2),     # groups of 64 experts (two 32-wide slots)
    (64, 6, "softmax", False, 2, 1),     # groups of 32
]


@pytest.mark.parametrize("cfg", CONFIGS, ids=[f"E{c[0]}k{c[1]}{c[2]}r{int(c[3])}g{c[4]}" for c in CONFIGS])
@pytest.mark.parametrize("M", [1, 7, 130])
def test_random_logits(cfg, M):
    E, k, scoring, renorm, ng, tg = cfg
    rng = np.random.default_rng(E * 1000 + M + k)
    _check(rng.standard_normal((M, E)) * 2.0, k, scoring, renorm, ng, tg)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("cfg", CONFIGS[:4])
def test_half_logits(cfg, dt):
    E, k, scoring, renorm, ng, tg = cfg
    rng = np.random.default_rng(E + k)
    _check(rng.standard_normal((257, E)) * 3.0, k, scoring, renorm, ng, tg, dt=dt)


@pytest.mark.parametrize("cfg", CONFIGS[:4] + CONFIGS[9:10] + CONFIGS[12:14])
def test_tied_logits(cfg):
    # integer logits: many exact ties, broken toward the lower index on both sides
    E, k, scoring, renorm, ng, tg = cfg
    rng = np.random.default_rng(11 + E)
    _check(rng.integers(-2, 3, size=(300, E)).astype(np.float64), k, scoring, renorm, ng, tg, max_ambiguous=1.0)


def test_non_finite_logits():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 64))
    x[0, :] = math.nan
    x[1, 3] = math.nan
    x[2, 7] = -math.inf
    x[3, :8] = -math.inf
    x[4, 9] = math.inf
    x[5, ::3] = math.nan
    for scoring, renorm in [("softmax", True), ("softmax", False), ("sigmoid", True), ("sigmoid", False)]:
        ids, _ = _check(x, 8, scoring, renorm)
        assert all(len(set(r)) == 8 for r in ids.tolist())
    _check(x, 8, "sigmoid", True, n_groups=8, topk_groups=2, max_ambiguous=0.05)
    _check(x, 8, "sigmoid", True, n_groups=2, topk_groups=1, max_ambiguous=0.05)  # groups of 32


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_workload_routing_full_size(name):
    # the workloads' own router logits at the largest M of their configs
    wl = WORKLOADS[name]
    M = 8192 if wl.E <= 64 else 4096
    logits = make_router_logits(wl, M, 77).numpy().astype(np.float64)
    r = routing_params(wl)
    _check(logits, wl.topk, r["scoring"], r["renormalize"], r["n_groups"], r["topk_groups"])


def test_feeds_align_and_layer_inputs():
    # the routing outputs are the align call's inputs as they are
    wl = WORKLOADS["deepseek_v3"]
    x = make_router_logits(wl, 64, 3).to(DEV)
    ids, _ = w.topk_routing(x, wl.topk, **routing_params(wl))
    s, e, npp, cnt = w.moe_align_block_size(ids, wl.E, 16)
    torch.cuda.synchronize()
    assert int(cnt.sum().item()) == 64 * wl.topk


def test_empty_batch_and_bad_arguments():
    x = torch.zeros(0, 64, device=DEV)
    ids, wt = w.topk_routing(x, 8)
    assert ids.shape == (0, 8) and wt.shape == (0, 8)
    with pytest.raises(w.WNA16Error):
        w.topk_routing(torch.zeros(4, 64, device=DEV), 8, "sigmoid", True, n_groups=8, topk_groups=0)
    with pytest.raises(ValueError):
        w.topk_routing(torch.zeros(4, 64, device=DEV, dtype=torch.float64), 8)


def test_graph_capture_replays():
    wl = WORKLOADS["deepseek_v3"]
    x = make_router_logits(wl, 128, 9).to(DEV)
    ids = torch.empty(128, wl.topk, dtype=torch.int32, device=DEV)
    wt = torch.empty(128, wl.topk, dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        w.topk_routing(x, wl.topk, topk_ids=ids, topk_weights=wt, stream=s, **routing_params(wl))
    torch.cuda.synchronize()
    ref = (ids.clone(), wt.clone())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        w.topk_routing(x, wl.topk, topk_ids=ids, topk_weights=wt, stream=s, **routing_params(wl))
    ids.zero_()
    wt.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(ids, ref[0]) and torch.equal(wt, ref[1])


@pytest.mark.parametrize("routing,E,k,ng,tg", [("softmax_renorm", 8, 2, 1, 1), ("softmax", 16, 4, 1, 1),
                                              ("sigmoid_grouped", 32, 4, 4, 2), ("sigmoid_grouped", 256, 8, 8, 4)])
@pytest.mark.parametrize("M", [1, 40, 128, 300])
def test_fused_layer_from_logits(routing, E, k, ng, tg, M):
    # one library call (routing, then the layer; up to 128 tokens routing and
    # align share one launch) = the two calls, bit for bit, and the oracle on
    # the oracle's routing
    from synthetic import Workload, make_layer_inputs
    from tests.helpers import bits_to_f64, halfbits, max_rel_err, oracle_layer_dict

    wl = Workload(name="routed", H=256, I=256, E=E, topk=k, bits=4, has_zeros=True, group_size=128,
                  act_dtype="f16", scale_dtype="f16", routing=routing, n_groups=ng, topk_groups=tg)
    li = make_layer_inputs(wl, M).to(DEV)
    logits = make_router_logits(wl, M, 5).to(DEV)
    rp = routing_params(wl)
    ids, wts = w.topk_routing(logits, k, **rp)
    y1 = w.fused_moe(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z, ids, wts, 4, 128)
    y2, ids2, wts2 = w.fused_moe_routed(li.hidden, li.w13_q, li.w13_s, li.w13_z, li.w2_q, li.w2_s, li.w2_z, logits,
                                        k, 4, 128, **rp)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids2) and torch.equal(wts, wts2) and torch.equal(y1, y2)
    # the routing against the oracle (near-tied group boundaries checked for
    # validity), then the layer against the oracle on the routing it ran
    _check(logits.double().cpu().numpy(), k, rp["scoring"], rp["renormalize"], rp["n_groups"], rp["topk_groups"])
    L = oracle_layer_dict(li)
    L["topk_ids"], L["topk_w"] = ids2.cpu().numpy(), wts2.cpu().numpy()
    ref = oracle.fused_moe_grouped(L)
    assert max_rel_err(bits_to_f64(halfbits(y2), "f16"), bits_to_f64(ref, "f16")) <= 1e-2
