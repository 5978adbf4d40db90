"""Each pin must have teeth: plant a plausible mistake in a copy of the oracle
(on the CPU) and check that at least one pin fails on it."""
import numpy as np
import pytest

import oracle
from oracle import moe_oracle as mo
import test_oracle_ffn as ffn_pins
import test_oracle_layout as layout_pins
import test_oracle_route as route_pins


def fails(pins, fn):
    for pin in pins:
        try:
            pin(fn)
        except (AssertionError, ValueError, IndexError):
            return True
    return False


def route_ties_to_higher_index(logits, k):
    L = np.asarray(logits, np.float32)
    E = L.shape[1]
    order = np.lexsort((-np.broadcast_to(np.arange(E), L.shape), -L.astype(np.float64)), axis=-1)
    ids = order[:, :k]
    sel = np.take_along_axis(L, ids, 1).astype(np.float64)
    z = np.exp(sel - sel.max(1, keepdims=True))
    return ids.astype(np.int32), z / z.sum(1, keepdims=True)


def route_softmax_over_all(logits, k):
    ids, _ = oracle.route(logits, k)
    L = np.asarray(logits, np.float64)
    p = np.exp(L - L.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    return ids, np.take_along_axis(p, ids.astype(np.int64), 1)


def route_sign_error(logits, k):
    ids, _ = oracle.route(logits, k)
    sel = np.take_along_axis(np.asarray(logits, np.float64), ids.astype(np.int64), 1)
    z = np.exp(sel.max(1, keepdims=True) - sel)
    return ids, z / z.sum(1, keepdims=True)


@pytest.mark.parametrize("mutant", [route_ties_to_higher_index, route_softmax_over_all,
                                    route_sign_error])
def test_route_mutants_are_caught(mutant):
    assert fails(route_pins.PINS, mutant)


_SWIGLU = mo.swiglu_mlp


def _swap_gate_up(X, wg, wu, wd):
    return _SWIGLU(X, wu, wg, wd)


def _silu_sign(X, wg, wu, wd):
    g, u = X @ wg.T, X @ wu.T
    h = g / (1.0 + np.exp(g)) * u
    return h, h @ wd.T


def _down_not_transposed(X, wg, wu, wd):
    g, u = X @ wg.T, X @ wu.T
    h = mo.silu(g) * u
    return h, h @ wd          # shape error unless square: wrong either way


@pytest.mark.parametrize("mutant", [_swap_gate_up, _silu_sign, _down_not_transposed])
def test_ffn_mutants_are_caught(mutant, monkeypatch):
    monkeypatch.setattr(mo, "swiglu_mlp", mutant)
    # the dense brute force shares swiglu_mlp, so use the pins that do not
    pins = [ffn_pins.check_single_expert_is_plain_swiglu, ffn_pins.check_two_experts_by_hand]
    assert fails(pins, mo.layer_forward)


def test_combine_dropping_a_term_is_caught(monkeypatch):
    def combine_missing_last(y, topk_w, pair_row, residual=None):
        w = np.array(topk_w, copy=True)
        w[:, -1] = 0.0
        return original(y, w, pair_row, residual)
    original = mo.combine
    monkeypatch.setattr(mo, "combine", combine_missing_last)
    assert fails([ffn_pins.check_dense_brute_force, ffn_pins.check_two_experts_by_hand],
                 mo.layer_forward)


def test_combine_without_residual_is_caught(monkeypatch):
    original = mo.combine
    monkeypatch.setattr(mo, "combine", lambda y, w, pr, residual=None: original(y, w, pr, None))
    assert fails([ffn_pins.check_zero_down_projection_leaves_residual], mo.layer_forward)


def layout_tokens_descending(ids, placement, E, W):
    lay = oracle.dispatch_layout(ids, placement, E, W)
    N, k = ids.shape
    # reverse the order of rows inside every expert segment
    rt = lay["row_token"].copy()
    pr = lay["pair_row"].copy()
    for e in range(E):
        a, n = lay["expert_offsets"][e], lay["expert_counts"][e]
        rt[a:a + n] = rt[a:a + n][::-1]
    for t in range(N):
        for j in range(k):
            e = ids[t, j]
            a, n = lay["expert_offsets"][e], lay["expert_counts"][e]
            pr[t, j] = a + (n - 1 - (lay["pair_row"][t, j] - a))
    lay["row_token"], lay["pair_row"] = rt, pr
    return lay


def layout_rank_by_expert_mod(ids, placement, E, W):
    """Plausible slip: rank(e) = e mod W instead of slot(e) // (E / W)."""
    fake = np.array([(e % W) * (E // W) + e // W for e in range(E)])
    inv = np.empty(E, np.int64)
    inv[fake] = np.arange(E)
    return oracle.dispatch_layout(ids, inv, E, W)


@pytest.mark.parametrize("mutant", [layout_tokens_descending, layout_rank_by_expert_mod])
def test_layout_mutants_are_caught(mutant):
    ids = layout_pins.random_ids(40, 8, 3, seed=9)
    with pytest.raises(AssertionError):
        layout_pins.check_invariants(mutant, ids, np.arange(8), 8, 4)


# ---- placement search and the router variants -----------------------------------------

import test_oracle_placement as placement_pins  # noqa: E402


def partition_without_gain_check(W, G, max_swaps):
    """Plausible slip: apply the best swap even when it does not improve."""
    W = np.asarray(W, dtype=np.int64)
    E = W.shape[0]
    group = np.arange(E) // (E // G)
    swaps = 0
    for _ in range(max_swaps):
        best, pair = None, None
        for a in range(E):
            for b in range(a + 1, E):
                if group[a] != group[b]:
                    g = mo.swap_gain(W, group, a, b)
                    if best is None or g > best:
                        best, pair = g, (a, b)
        if pair is None or swaps >= 3 * E:
            break
        a, b = pair
        group[a], group[b] = group[b], group[a]
        swaps += 1
    return group, swaps


def swap_gain_sign_error(W, group, a, b):
    return -_SWAP_GAIN(W, group, a, b)


_SWAP_GAIN = mo.swap_gain


@pytest.mark.parametrize("mutant,target", [(partition_without_gain_check, "partition"),
                                           (swap_gain_sign_error, "swap_gain")])
def test_placement_mutants_are_caught(mutant, target, monkeypatch):
    monkeypatch.setattr(mo, target, mutant)
    monkeypatch.setattr(oracle, target, mutant)
    pins = [lambda: placement_pins.test_partition_is_balanced_and_locally_optimal(12, 3, 4),
            placement_pins.test_swap_gain_is_the_change_of_the_objective,
            placement_pins.test_ties_take_the_first_pair_in_lexicographic_order]
    caught = False
    for pin in pins:
        try:
            pin()
        except AssertionError:
            caught = True
            break
    assert caught


def test_sigmoid_router_mutant_with_biased_weights_is_caught(monkeypatch):
    """Slip: the weights renormalise s + bias instead of s."""
    original = mo.route_sigmoid_bias

    def mutant(logits, bias, k):
        ids, _ = original(logits, bias, k)
        L = np.asarray(logits, np.float64)
        s = 1.0 / (1.0 + np.exp(-L)) + np.asarray(bias, np.float64)[None, :]
        sel = np.take_along_axis(s, ids.astype(np.int64), 1)
        return ids, sel / sel.sum(1, keepdims=True)

    monkeypatch.setattr(oracle, "route_sigmoid_bias", mutant)
    with pytest.raises(AssertionError):
        route_pins.test_sigmoid_bias_router_pins()


# ---- bf16 widening and the Table I counters ------------------------------------------

import test_oracle_helpers as helper_pins  # noqa: E402


def widen_shift_15(a):
    """Slip: shift by 15 instead of 16."""
    a = np.asarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 15).view(np.float32).astype(np.float64)


def widen_drops_sign(a):
    """Slip: the sign bit masked off."""
    a = np.asarray(a, dtype=np.uint16) & np.uint16(0x7FFF)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def widen_nan_to_zero(a):
    """Slip: non-finite patterns flushed to zero."""
    v = oracle.widen_bf16(a)
    return np.where(np.isfinite(v), v, 0.0)


def widen_as_fp16(a):
    """Slip: the bits read as IEEE half precision instead of bfloat16."""
    return np.asarray(a, dtype=np.uint16).view(np.float16).astype(np.float64)


def widen_low_half(a):
    """Slip: the pattern put in the low half of the binary32 word."""
    return np.asarray(a, dtype=np.uint16).astype(np.uint32).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("mutant", [widen_shift_15, widen_drops_sign, widen_nan_to_zero,
                                    widen_as_fp16, widen_low_half])
def test_widen_mutants_are_caught(mutant):
    assert fails(helper_pins.WIDEN_PINS, mutant)


def stats_share_counts_two_ranks(layout, N, k, W):
    s = oracle.layout_stats(layout, N, k, W)
    distinct = layout["rank_member"].sum(axis=1)
    s["same_rank_share"] = float(np.mean(distinct <= 2))
    return s


def stats_ranks_over_rows(layout, N, k, W):
    """Slip: distinct ranks divided by rows instead of tokens."""
    s = oracle.layout_stats(layout, N, k, W)
    s["ranks_per_token"] = layout["n_dedup_rows"] / (N * k)
    return s


def stats_reduction_inverted(layout, N, k, W):
    s = oracle.layout_stats(layout, N, k, W)
    s["dedup_reduction"] = layout["n_dedup_rows"] / (N * k)
    return s


def stats_load_over_max(layout, N, k, W):
    """Slip: the mean load taken over the ranks instead of the experts."""
    s = oracle.layout_stats(layout, N, k, W)
    s["max_over_mean_load"] = float(layout["expert_counts"].max() / (N * k / W))
    return s


@pytest.mark.parametrize("mutant", [stats_share_counts_two_ranks, stats_ranks_over_rows,
                                    stats_reduction_inverted, stats_load_over_max])
def test_layout_stats_mutants_are_caught(mutant):
    assert fails(helper_pins.STATS_PINS, mutant)
