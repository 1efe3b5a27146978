"""Pins for the oracle's router: the GLM-5.2 write-up's router check re-run as data,
brute-force enumeration of group and expert subsets, closed forms."""
import itertools
import json
import math
import os
from types import SimpleNamespace

import numpy as np
import pytest

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def cfg(G, tg, k, rsf=1.0):
    return SimpleNamespace(n_groups=G, topk_group=tg, top_k=k, routed_scaling_factor=rsf)


def test_writeup_router_cases():
    gold = json.load(open(os.path.join(GOLD, "router_glm52_writeup_cases.json")))
    for c in gold["cases"]:
        idx, w = oracle.route(np.array([c["logits"]]), np.array(c["bias"], np.float32),
                              cfg(1, 1, c["top_k"]))
        assert int(idx[0, -1]) == c["last"], c["name"]
        if "selected_set" in c:
            assert sorted(idx[0].tolist()) == c["selected_set"]
        assert math.isclose(w.sum(), 1.0, rel_tol=1e-12)
    if gold["rejects_nonfinite"]:
        rng = np.random.default_rng(5)
        logits = rng.normal(size=(64, 256))
        logits[3, 17] = np.nan
        with pytest.raises(ValueError):
            oracle.route(logits, np.zeros(256, np.float32), cfg(1, 1, 8))
        with pytest.raises(ValueError):
            b = np.zeros(256, np.float32)
            b[0] = np.inf
            oracle.route(np.zeros((1, 256)), b, cfg(1, 1, 8))


def _brute(c_row, G, tg, k):
    """Enumerate every kept-group subset and every k-subset of its experts."""
    E = len(c_row)
    size = E // G
    gscore = []
    for g in range(G):
        vals = sorted(c_row[g * size:(g + 1) * size], reverse=True)
        gscore.append(sum(vals[:min(2, size)]))
    best_groups = max(itertools.combinations(range(G), tg),
                      key=lambda gs: sum(gscore[g] for g in gs))
    cand = [e for g in best_groups for e in range(g * size, (g + 1) * size)]
    best = max(itertools.combinations(cand, k), key=lambda es: sum(c_row[e] for e in es))
    return sorted(best, key=lambda e: -c_row[e])


@pytest.mark.parametrize("E,G,tg,k", [(16, 4, 2, 4), (12, 3, 2, 3), (8, 2, 1, 2), (8, 8, 3, 3),
                                      (16, 1, 1, 5), (6, 3, 3, 6)])
def test_route_matches_brute_force(E, G, tg, k):
    rng = np.random.default_rng(E * 100 + G * 10 + k)
    logits = rng.normal(size=(40, E))
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    c = cfg(G, tg, k, 2.5)
    idx, w = oracle.route(logits, bias, c)
    marg = oracle.route_margins(logits, bias, c)
    s = 1.0 / (1.0 + np.exp(-logits))
    cc = s + bias.astype(np.float64)
    for t in range(logits.shape[0]):
        if marg[t] < 1e-9:
            continue
        assert idx[t].tolist() == _brute(cc[t], G, tg, k)
    assert np.allclose(w.sum(axis=1), 2.5, rtol=1e-12)


def test_single_group_is_plain_topk():
    # with one group the router is the plain sigmoid top-k of the write-up's check:
    # full order by (-score, id)
    rng = np.random.default_rng(7)
    logits = rng.normal(size=(64, 256))
    bias = rng.normal(scale=0.05, size=256).astype(np.float32)
    idx, _ = oracle.route(logits, bias, cfg(1, 1, 8))
    score = 1.0 / (1.0 + np.exp(-logits)) + bias.astype(np.float64)
    for t in range(64):
        order = np.lexsort((np.arange(256), -score[t]))[:8]
        assert idx[t].tolist() == order.tolist()


def test_gate_weights_closed_forms():
    # all logits 0: every affinity is 0.5, so each weight is rsf/k whatever the bias
    bias = np.array([0.3, -0.2, 0.1, 0.0, 0.05, -0.1, 0.2, -0.3], np.float32)
    idx, w = oracle.route(np.zeros((1, 8)), bias, cfg(2, 1, 3, 2.5))
    assert np.allclose(w, 2.5 / 3, rtol=1e-14)
    # two experts with affinities 3/4 and 1/2: weights 0.6 and 0.4 (x rsf)
    idx, w = oracle.route(np.array([[math.log(3.0), 0.0, -5.0, -5.0]]),
                          np.zeros(4, np.float32), cfg(1, 1, 2, 2.5))
    assert idx[0].tolist() == [0, 1]
    assert np.allclose(w[0], [1.5, 1.0], rtol=1e-14)


def test_bias_ranks_only():
    # bias moves expert 3 into the selection, but weights use unbiased affinities
    logits = np.array([[2.0, 1.0, 0.5, 0.0]])
    idx, w = oracle.route(logits, np.array([0, 0, 0, 0.9], np.float32), cfg(1, 1, 2, 1.0))
    assert idx[0].tolist() == [3, 0]
    s = np.array([0.5, 1.0 / (1.0 + math.exp(-2.0))])
    assert np.allclose(w[0], s / s.sum(), rtol=1e-14)


def test_dropped_groups_never_selectable():
    # group 0 = experts {0,1}, group 1 = {2,3}; scores c = [0.5, 0.45, 0.9, -0.5]
    # group sums 0.95 vs 0.4 keep group 0 although expert 2 has the best score
    bias = np.array([0.0, -0.05, 0.4, -1.0], np.float32)
    idx, _ = oracle.route(np.zeros((1, 4)), bias, cfg(2, 1, 2))
    assert idx[0].tolist() == [0, 1]
    # kept experts with negative scores still win over dropped ones: masking
    # dropped experts to 0 instead of -inf would pick experts 2 and 3 here
    bias = np.array([-0.6, -0.7, -0.2, -1.4], np.float32)   # c = [-0.1,-0.2,0.3,-0.9]
    idx, _ = oracle.route(np.zeros((1, 4)), bias, cfg(2, 1, 2))
    assert idx[0].tolist() == [0, 1]
    bias = np.array([0.1, 0.1, -0.3, -0.5], np.float32)     # c = [0.6,0.6,0.2,0.0]
    idx, _ = oracle.route(np.zeros((1, 4)), bias, cfg(2, 1, 2))
    assert idx[0].tolist() == [0, 1]


def test_group_ties_go_to_lower_group():
    idx, _ = oracle.route(np.zeros((1, 8)), np.zeros(8, np.float32), cfg(4, 2, 2))
    assert idx[0].tolist() == [0, 1]


def test_margins():
    logits = np.array([[1.0, 1.0, 1.0, 1.0, 0.3, 0.29999, -1.0, -1.0]])
    m = oracle.route_margins(logits, np.zeros(8, np.float32), cfg(1, 1, 5))
    s = 1.0 / (1.0 + np.exp(-logits[0]))
    assert m[0] == 0.0  # experts 0..3 tie exactly
    m2 = oracle.route_margins(np.array([[4.0, 3.0, 2.0, 1.0, 0.0]]), np.zeros(5, np.float32), cfg(1, 1, 2))
    s = 1.0 / (1.0 + np.exp(-np.array([4.0, 3.0, 2.0])))
    assert math.isclose(m2[0], min(s[0] - s[1], s[1] - s[2]), rel_tol=1e-12)


def test_config_validation():
    with pytest.raises(ValueError):
        oracle.route(np.zeros((1, 10)), np.zeros(10, np.float32), cfg(3, 1, 2))
    with pytest.raises(ValueError):
        oracle.route(np.zeros((1, 8)), np.zeros(8, np.float32), cfg(4, 1, 3))


def test_designed_exact_ties_select_as_derived_by_hand():
    """The tie designs used by the GPU tie tests: the oracle's selection on
    them is the one derived by hand from the lower-id rule (GLM-5.2 write-up,
    'How it works (validated core mechanics)'), and the gate weights are
    exactly rsf / k (every selected affinity is 1/2)."""
    from helpers import tie_design
    for shape in (synth.TINY, synth.GLM):
        bias, expect = tie_design(shape)
        logits = np.zeros((3, shape.n_experts))
        idx, w = oracle.route(logits, bias, shape)
        assert idx.tolist() == [expect] * 3
        assert np.all(w == shape.routed_scaling_factor / shape.top_k)
        # the bias values sit on the 2^-10 grid: 1/2 + b is exact in fp32
        c32 = np.float32(0.5) + bias
        assert np.array_equal(c32.astype(np.float64), 0.5 + bias.astype(np.float64))


def test_duplicated_group_ties_go_to_the_lower_id():
    from helpers import duplicate_group, route_margins_except_exact
    shape = synth.TINY
    wr, b = duplicate_group(synth.router_weight(shape, 4), synth.router_bias(shape, 4), shape, 0, 1)
    x = synth.token_batch(shape, 4, "dup", range(40))
    idx, _ = oracle.route(oracle.router_logits(x, wr), b, shape)
    both = 0
    for row in idx:
        for e in row:
            if e < 4:      # an expert of group 0 selected ...
                if e + 4 in row:   # ... with its twin: the lower id comes first
                    both += 1
                    assert list(row).index(e) < list(row).index(e + 4)
            if 4 <= e < 8:         # a group-1 expert only with its group-0 twin before it
                assert e - 4 in row and list(row).index(e - 4) < list(row).index(e)
    assert both > 0
    assert np.all(route_margins_except_exact(oracle.router_logits(x, wr), b, shape) > 0)
