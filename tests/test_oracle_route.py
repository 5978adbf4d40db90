"""Pins of the oracle's router against definitions it does not use itself.

The router keeps the k largest fp32 logits (ties to the lower expert index) and
weights them by a softmax over the selected k ("Expert Coupling", Appendix
A-A1 Table II; FarSkip-Collective Sec. 2.1).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
from combine_warp_top_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def selected_by_definition(L, k):
    """Expert e is selected iff fewer than k experts beat it, where e' beats e
    when L[e'] > L[e], or L[e'] == L[e] and e' < e.  Returned in the order
    of the beat relation (best first)."""
    E = len(L)
    beats = [sum(1 for f in range(E) if L[f] > L[e] or (L[f] == L[e] and f < e)) for e in range(E)]
    chosen = [e for e in range(E) if beats[e] < k]
    return sorted(chosen, key=lambda e: beats[e])


def check_route_brute_force(route_fn):
    rng = np.random.default_rng(1)
    for trial in range(200):
        E = int(rng.integers(1, 9))
        k = int(rng.integers(1, E + 1))
        # coarse values so that ties are frequent
        L = rng.integers(-3, 4, size=(1, E)).astype(np.float32) * np.float32(0.5)
        ids, w = route_fn(L, k)
        assert ids[0].tolist() == selected_by_definition(L[0].tolist(), k), (L, k, ids)
    # many experts and up to the largest k the library accepts
    for trial in range(40):
        E = int(rng.integers(24, 65))
        k = int(rng.integers(8, min(E, 32) + 1))
        L = rng.integers(-4, 5, size=(1, E)).astype(np.float32) * np.float32(0.25)
        ids, w = route_fn(L, k)
        assert ids[0].tolist() == selected_by_definition(L[0].tolist(), k), (L, k, ids)


def check_subset_sum_is_max(route_fn):
    """With distinct logits the selected set is the k-subset of largest sum."""
    rng = np.random.default_rng(2)
    for trial in range(50):
        E, k = 7, int(rng.integers(1, 5))
        L = rng.standard_normal((1, E)).astype(np.float32)
        best = max(itertools.combinations(range(E), k), key=lambda s: sum(float(L[0, e]) for e in s))
        ids, _ = route_fn(L, k)
        assert set(ids[0].tolist()) == set(best)


def check_k2_closed_form(route_fn):
    """k = 2: w_1 = 1 / (1 + exp(L_2 - L_1)), w_2 = 1 - w_1."""
    L = synth.normal_f32(0, 11, (300, 10))
    ids, w = route_fn(L, 2)
    L1 = np.take_along_axis(L, ids[:, :1].astype(np.int64), 1)[:, 0].astype(np.float64)
    L2 = np.take_along_axis(L, ids[:, 1:].astype(np.int64), 1)[:, 0].astype(np.float64)
    w1 = 1.0 / (1.0 + np.exp(L2 - L1))
    np.testing.assert_allclose(w[:, 0], w1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(w[:, 1], 1.0 - w1, rtol=0, atol=1e-12)


def check_weights_sum_to_one(route_fn):
    L = synth.normal_f32(0, 12, (500, 16))
    for k in (1, 3, 8, 16):
        _, w = route_fn(L, k)
        np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-12)
        assert np.all(np.diff(w, axis=1) <= 1e-15), "weights follow the descending logit order"


def check_ties(route_fn):
    # all equal: the first k experts, uniform weights
    L = np.zeros((3, 8), np.float32)
    ids, w = route_fn(L, 3)
    assert ids.tolist() == [[0, 1, 2]] * 3
    np.testing.assert_allclose(w, 1.0 / 3.0, atol=1e-15)
    # a tie straddling the cut: the lower index wins
    L = np.array([[0.0, 1.0, 0.5, 1.0, 0.5]], np.float32)
    ids, _ = route_fn(L, 3)
    assert ids.tolist() == [[1, 3, 2]]
    # +0.0 and -0.0 compare equal: index decides
    L = np.array([[-0.0, 0.0, -1.0]], np.float32)
    ids, _ = route_fn(L, 1)
    assert ids.tolist() == [[0]]


def check_softmax_matches_full_softmax_ratio(route_fn):
    """The selected weights are the full-softmax probabilities renormalised over
    the selected k ("softmax over all E, then top-k" of Table II, renormalised):
    the ratios w_i / w_j equal exp(L_i - L_j) under both readings."""
    L = synth.normal_f32(0, 13, (200, 12))
    ids, w = route_fn(L, 4)
    Lf = L.astype(np.float64)
    p = np.exp(Lf - Lf.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    ps = np.take_along_axis(p, ids.astype(np.int64), 1)
    np.testing.assert_allclose(w, ps / ps.sum(1, keepdims=True), rtol=1e-12)


PINS = [check_route_brute_force, check_subset_sum_is_max, check_k2_closed_form,
        check_weights_sum_to_one, check_ties, check_softmax_matches_full_softmax_ratio]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_route_pins(pin):
    pin(oracle.route)


def test_worked_example_routing_and_receivers():
    """The pages' W=3, top-2 example: A->{E0,E2}, B->{E1,E2}, C->{E0,E1};
    each rank holds one expert and receives P0:{A,C}, P1:{B,C}, P2:{A,B}."""
    g = json.load(open(os.path.join(GOLDEN, "worked_routing_example.json")))
    toks = g["tokens"]
    # logits that realise the table: the two routed experts score above the third
    L = np.full((3, 3), -1.0, np.float32)
    for t, name in enumerate(toks):
        for rank_in_choice, e in enumerate(g["routing"][name]):
            L[t, e] = 2.0 - rank_in_choice
    ids, w = oracle.route(L, g["k"])
    for t, name in enumerate(toks):
        assert sorted(ids[t].tolist()) == sorted(g["routing"][name])
    lay = oracle.dispatch_layout(ids, np.arange(3), g["E"], g["W"])
    for r in range(g["W"]):
        a, b = lay["rank_offsets"][r], lay["rank_offsets"][r + 1]
        got = [toks[t] for t in lay["row_token"][a:b]]
        assert got == g["received_by_rank"][str(r)]
    assert lay["expert_counts"].tolist() == [2, 2, 2]
    assert lay["n_dedup_rows"] == 6  # one expert per rank: nothing to merge
    # dedup rows are the same receive sets
    for r in range(g["W"]):
        a, b = lay["dedup_offsets"][r], lay["dedup_offsets"][r + 1]
        assert [toks[t] for t in lay["dedup_row_token"][a:b]] == g["received_by_rank"][str(r)]


def test_route_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.route(np.zeros((2, 4), np.float32), 5)
    with pytest.raises(ValueError):
        oracle.route(np.array([[np.nan, 1.0]], np.float32), 1)


def test_full_softmax_variant():
    """renormalize=False: the same experts, weighted by their probability under
    the softmax over all E (closed form for E = 2, k = 1: 1 / (1 + e^{L_2 - L_1}))."""
    L = synth.normal_f32(0, 14, (300, 2))
    ids, w = oracle.route(L, 1, renormalize=False)
    Lsel = np.take_along_axis(L, ids.astype(np.int64), 1)[:, 0].astype(np.float64)
    Loth = np.take_along_axis(L, 1 - ids.astype(np.int64), 1)[:, 0].astype(np.float64)
    np.testing.assert_allclose(w[:, 0], 1.0 / (1.0 + np.exp(Loth - Lsel)), atol=1e-12)
    L = synth.normal_f32(0, 15, (200, 16))
    ids_r, w_r = oracle.route(L, 4)
    ids_f, w_f = oracle.route(L, 4, renormalize=False)
    assert np.array_equal(ids_r, ids_f)
    assert np.all(w_f.sum(1) < 1.0)
    np.testing.assert_allclose(w_f / w_f.sum(1, keepdims=True), w_r, rtol=1e-12)
    ids_all, w_all = oracle.route(L, 16, renormalize=False)
    np.testing.assert_allclose(w_all.sum(1), 1.0, atol=1e-12)  # k = E: all probabilities


def test_sigmoid_bias_router_pins():
    """The aux-loss-free sigmoid router: selection by fp32(sigmoid(L)) + bias
    (brute force by definition), weights = selected scores renormalised, bias
    steering the choice but not the weights."""
    rng = np.random.default_rng(5)
    for trial in range(100):
        E = int(rng.integers(2, 12))
        k = int(rng.integers(1, E + 1))
        L = (rng.integers(-8, 9, size=(1, E)) * 0.25).astype(np.float32)
        b = (rng.integers(-3, 4, size=E) * 0.05).astype(np.float32)
        ids, w = oracle.route_sigmoid_bias(L, b, k)
        s = (1.0 / (1.0 + np.exp(-L[0].astype(np.float64)))).astype(np.float32)
        key = (s + b).astype(np.float32)
        assert ids[0].tolist() == selected_by_definition(key.tolist(), k)
        sel = s[ids[0]].astype(np.float64)
        np.testing.assert_allclose(w[0], sel / sel.sum(), rtol=1e-15)
    # zero bias and well separated logits: the same experts as the softmax router
    L = (rng.permuted(np.tile(np.arange(16), (50, 1)), axis=1) * 0.3 - 2.0).astype(np.float32)
    ids_s, _ = oracle.route_sigmoid_bias(L, np.zeros(16, np.float32), 4)
    ids_r, _ = oracle.route(L, 4)
    assert np.array_equal(ids_s, ids_r)
    # a large bias forces the choice; the weights still come from the scores alone
    L = synth.normal_f32(0, 16, (20, 8))
    b = np.zeros(8, np.float32)
    b[[1, 6]] = 10.0
    ids, w = oracle.route_sigmoid_bias(L, b, 2)
    assert all(sorted(r) == [1, 6] for r in ids.tolist())
    s = 1.0 / (1.0 + np.exp(-L.astype(np.float64)))
    for t in range(20):
        a, c = ids[t]
        np.testing.assert_allclose(w[t], [s[t, a] / (s[t, a] + s[t, c]), s[t, c] / (s[t, a] + s[t, c])],
                                   rtol=1e-7)
