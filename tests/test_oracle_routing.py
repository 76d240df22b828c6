"""Pins of the oracle's top-k routing (CPU only).

The oracle's routing is checked against closed forms worked by hand, brute
force over all expert subsets on tiny inputs, invariants, and the torch-based
router of the synthetic workloads (an independent implementation of the same
readings).
"""
import itertools
import math

import numpy as np
import pytest

import oracle
from synthetic import WORKLOADS, make_router_logits, make_routing, routing_params


def _logit(p):
    p = np.asarray(p, dtype=np.float64)
    return np.log(p / (1.0 - p))


def test_softmax_closed_form():
    # softmax of log(1..4) is (0.1, 0.2, 0.3, 0.4)
    l = np.log(np.array([[1.0, 2.0, 3.0, 4.0]]))
    ids, w = oracle.topk_routing(l, 2, "softmax", renormalize=False)
    assert ids.tolist() == [[3, 2]]
    np.testing.assert_allclose(w, [[0.4, 0.3]], rtol=1e-14)
    ids, w = oracle.topk_routing(l, 2, "softmax", renormalize=True)
    assert ids.tolist() == [[3, 2]]
    np.testing.assert_allclose(w, [[4 / 7, 3 / 7]], rtol=1e-14)


def test_sigmoid_grouped_closed_form():
    # scores p (logits = logit(p)); groups of 2: sums 1.0, 1.1, 0.9, 1.1 -> keep
    # groups 1 and 3 -> experts {2, 3, 6, 7} with scores .5 .6 .3 .8 -> top-2 = 7, 3
    p = np.array([[0.1, 0.9, 0.5, 0.6, 0.7, 0.2, 0.3, 0.8]])
    l = _logit(p)
    np.testing.assert_allclose(oracle.routing_group_scores(l, "sigmoid", 4), [[1.0, 1.1, 0.9, 1.1]], rtol=1e-14)
    ids, w = oracle.topk_routing(l, 2, "sigmoid", renormalize=True, n_groups=4, topk_groups=2)
    assert ids.tolist() == [[7, 3]]
    np.testing.assert_allclose(w, [[0.8 / 1.4, 0.6 / 1.4]], rtol=1e-13)
    # expert 1 (0.9) is the best overall but its group (1.0) is dropped
    ids, _ = oracle.topk_routing(l, 1, "sigmoid", renormalize=False, n_groups=1)
    assert ids.tolist() == [[1]]
    ids, w = oracle.topk_routing(l, 1, "sigmoid", renormalize=False, n_groups=4, topk_groups=2)
    assert ids.tolist() == [[7]]
    np.testing.assert_allclose(w, [[0.8]], rtol=1e-14)


def test_group_score_is_two_best_not_max():
    # group 0 holds the best single expert (0.95) but the worse pair (0.95 + 0.05);
    # group 1's pair .6 + .6 wins with one group kept
    l = _logit(np.array([[0.95, 0.05, 0.6, 0.6]]))
    ids, _ = oracle.topk_routing(l, 1, "sigmoid", renormalize=True, n_groups=2, topk_groups=1)
    assert ids.tolist() == [[2]]


def test_ties_go_to_the_lower_index():
    l = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]])
    ids, w = oracle.topk_routing(l, 3, "softmax", renormalize=True)
    assert ids.tolist() == [[1, 2, 4]]
    np.testing.assert_allclose(w, [[1 / 3, 1 / 3, 1 / 3]], rtol=1e-14)
    # tied group scores: the lower group is kept
    l = np.array([[0.0, 1.0, 1.0, 0.0, 2.0, -5.0]])
    ids, _ = oracle.topk_routing(l, 2, "sigmoid", renormalize=True, n_groups=3, topk_groups=1)
    assert ids.tolist() == [[1, 0]]


def test_nan_ranks_as_minus_infinity():
    l = np.array([[-math.inf, 0.0, math.nan, 1.0, -7.0]])
    ids, _ = oracle.topk_routing(l, 5, "sigmoid", renormalize=False)
    assert ids.tolist() == [[3, 1, 4, 0, 2]]


def _brute_topk(scores, allowed, k):
    best = max(itertools.combinations(allowed, k), key=lambda c: sum(scores[e] for e in c))
    return sorted(best, key=lambda e: -scores[e])


@pytest.mark.parametrize("seed", range(24))
def test_random_vs_brute_force(seed):
    rng = np.random.default_rng(seed)
    n_groups = [1, 2, 3, 4][seed % 4]
    gs = int(rng.integers(2, 4))
    E = n_groups * gs
    topk_groups = int(rng.integers(1, n_groups + 1))
    k = int(rng.integers(1, min(3, topk_groups * gs) + 1))
    scoring = "softmax" if seed % 2 else "sigmoid"
    renorm = bool((seed // 2) % 2)
    l = rng.standard_normal((3, E))
    ids, w = oracle.topk_routing(l, k, scoring, renorm, n_groups, topk_groups)
    for t in range(l.shape[0]):
        if scoring == "softmax":
            sc = np.exp(l[t]) / np.exp(l[t]).sum()
        else:
            sc = np.array([1.0 / (1.0 + math.exp(-v)) for v in l[t]])
        allowed = list(range(E))
        if n_groups > 1:
            # group score: the best pair sum inside the group, by enumeration
            gsc = [max(sc[a] + sc[b] for a, b in itertools.combinations(range(g * gs, (g + 1) * gs), 2))
                   for g in range(n_groups)]
            kept = max(itertools.combinations(range(n_groups), topk_groups), key=lambda c: sum(gsc[g] for g in c))
            allowed = [e for g in kept for e in range(g * gs, (g + 1) * gs)]
        want = _brute_topk(sc, allowed, k)
        assert ids[t].tolist() == want
        exp_w = sc[want] / sc[want].sum() if renorm else sc[want]
        np.testing.assert_allclose(w[t], exp_w, rtol=1e-12)


def test_invariants():
    rng = np.random.default_rng(7)
    l = rng.standard_normal((50, 64)) * 2
    for scoring in ("softmax", "sigmoid"):
        ids, w = oracle.topk_routing(l, 6, scoring, renormalize=True, n_groups=8, topk_groups=3)
        np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-13)
        assert all(len(set(r)) == 6 for r in ids.tolist())
        # at most topk_groups distinct groups
        assert max(len(set((r // 8).tolist())) for r in ids) <= 3
        # keeping every group is plain top-k
        a = oracle.topk_routing(l, 6, scoring, True, n_groups=8, topk_groups=8)
        b = oracle.topk_routing(l, 6, scoring, True, n_groups=1, topk_groups=1)
        assert (a[0] == b[0]).all()
        np.testing.assert_allclose(a[1], b[1], rtol=1e-14)
    # weights descend along the slots
    ids, w = oracle.topk_routing(l, 8, "softmax", renormalize=False)
    assert (np.diff(w, axis=1) <= 0).all()
    # k = E selects every expert
    ids, w = oracle.topk_routing(l[:, :8], 8, "sigmoid", renormalize=True)
    assert (np.sort(ids, 1) == np.arange(8)).all()


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_agrees_with_workload_router(name):
    wl = WORKLOADS[name]
    M = 64
    logits = make_router_logits(wl, M, 123).numpy()
    ids_ref, w_ref = make_routing(wl, M, 123)
    ids, w = oracle.topk_routing(logits, wl.topk, **routing_params(wl))
    assert (ids == ids_ref.numpy()).all()
    np.testing.assert_allclose(w, w_ref.numpy(), rtol=1e-6, atol=1e-7)
