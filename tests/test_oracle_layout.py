"""Pins of the oracle's dispatch layout (plain and deduplicated).

Sources: "Kernel fusion for expert parallelism", section "Expert parallelism:
dispatch and combine" (E/W experts per rank; a token whose experts lie on d
ranks leaves its owner d <= min(k, W) times) and section "INC all-to-all
phased" (the W_x estimate); "Expert Coupling" Sec. II-B Table I (distinct
GPUs per token and deduplication share under contiguous placement) and Sec.
V-A (one row per unique (token, rank); placement is a permutation of expert
IDs and does not change routing).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from combine_warp_top_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def expected_distinct_ranks(E, W, k):
    """Uniform routing without replacement: a rank of E/W experts is missed with
    probability C(E - E/W, k) / C(E, k)."""
    return W * (1.0 - math.comb(E - E // W, k) / math.comb(E, k))


def expected_same_rank_share(E, W, k):
    return W * math.comb(E // W, k) / math.comb(E, k)


def random_ids(N, E, k, seed):
    L = synth.normal_f32(seed, 21, (N, E))
    ids, _ = oracle.route(L, k)
    return ids


def check_invariants(layout_fn, ids, placement, E, W):
    N, k = ids.shape
    lay = layout_fn(ids, placement, E, W)
    R = N * k
    slot = np.empty(E, np.int64)
    slot[np.asarray(placement)] = np.arange(E)
    rank = slot // (E // W)
    # counts and offsets
    assert lay["expert_counts"].sum() == R
    assert np.array_equal(lay["expert_counts"], np.bincount(ids.reshape(-1), minlength=E))
    assert lay["expert_offsets"][E] == R
    for p in range(E):  # segments are laid out in slot order, back to back
        e = placement[p]
        nxt = lay["expert_offsets"][placement[p + 1]] if p + 1 < E else R
        assert lay["expert_offsets"][e] + lay["expert_counts"][e] == nxt
    assert lay["rank_offsets"][0] == 0 and lay["rank_offsets"][W] == R
    # every (token, expert) pair appears exactly once, at pair_row
    row_token, pair_row = lay["row_token"], lay["pair_row"]
    assert sorted(pair_row.reshape(-1).tolist()) == list(range(R))
    for t in range(N):
        for j in range(k):
            i = pair_row[t, j]
            e = ids[t, j]
            assert row_token[i] == t
            assert lay["expert_offsets"][e] <= i < lay["expert_offsets"][e] + lay["expert_counts"][e]
    # tokens ascend inside each expert segment
    for e in range(E):
        a = lay["expert_offsets"][e]
        seg = row_token[a:a + lay["expert_counts"][e]]
        assert np.all(np.diff(seg) > 0)
    # rank slices hold exactly the rows of that rank's experts
    for r in range(W):
        a, b = lay["rank_offsets"][r], lay["rank_offsets"][r + 1]
        for i in range(a, b):
            t = row_token[i]
            js = np.nonzero(pair_row[t] == i)[0]
            assert len(js) == 1 and rank[ids[t, js[0]]] == r
    # dedup: one row per distinct (token, rank)
    distinct = {(t, int(rank[e])) for t in range(N) for e in ids[t]}
    R_d = lay["n_dedup_rows"]
    assert R_d == len(distinct)
    assert N <= R_d <= N * min(k, W)
    got = set()
    for r in range(W):
        a, b = lay["dedup_offsets"][r], lay["dedup_offsets"][r + 1]
        toks = lay["dedup_row_token"][a:b]
        assert np.all(np.diff(toks) > 0)
        got |= {(int(t), r) for t in toks}
    assert got == distinct
    for t in range(N):
        for j in range(k):
            d = lay["pair_dedup_row"][t, j]
            r = int(rank[ids[t, j]])
            assert lay["dedup_row_token"][d] == t
            assert lay["dedup_offsets"][r] <= d < lay["dedup_offsets"][r + 1]
            assert lay["expand_src"][pair_row[t, j]] == d
    return lay


@pytest.mark.parametrize("N,E,k,W", [(50, 8, 2, 2), (40, 16, 4, 4), (30, 6, 6, 3), (33, 8, 3, 8),
                                     (25, 8, 8, 1), (64, 12, 1, 4), (40, 24, 12, 6),
                                     (20, 64, 32, 16)])
def test_layout_invariants(N, E, k, W):
    ids = random_ids(N, E, k, seed=N + E)
    check_invariants(oracle.dispatch_layout, ids, np.arange(E), E, W)


def test_layout_invariants_permuted_placement():
    E, W, k, N = 12, 4, 3, 60
    ids = random_ids(N, E, k, seed=5)
    placement = synth.permutation(0, 31, E).astype(np.int32)
    lay = check_invariants(oracle.dispatch_layout, ids, placement, E, W)
    plain = oracle.dispatch_layout(ids, np.arange(E), E, W)
    # placement changes where rows live, never which (token, expert) pairs exist
    assert np.array_equal(np.sort(lay["expert_counts"]), np.sort(plain["expert_counts"]))


def test_one_expert_per_rank_has_nothing_to_merge():
    ids = random_ids(200, 8, 2, seed=3)
    lay = oracle.dispatch_layout(ids, np.arange(8), 8, 8)
    assert lay["n_dedup_rows"] == 200 * 2


def test_single_rank_merges_to_one_row_per_token():
    ids = random_ids(100, 8, 4, seed=4)
    lay = oracle.dispatch_layout(ids, np.arange(8), 8, 1)
    assert lay["n_dedup_rows"] == 100
    assert np.array_equal(lay["dedup_row_token"], np.arange(100))


def test_all_tokens_on_one_expert():
    N, E, k = 20, 8, 1
    ids = np.full((N, k), 5, np.int32)
    lay = oracle.dispatch_layout(ids, np.arange(E), E, 4)
    assert lay["expert_counts"].tolist() == [0] * 5 + [N] + [0] * 2
    assert np.array_equal(lay["row_token"], np.arange(N))


def test_bad_placement_rejected():
    with pytest.raises(ValueError):
        oracle.dispatch_layout(np.zeros((2, 1), np.int32), np.array([0, 0, 1, 2]), 4, 2)
    with pytest.raises(ValueError):
        oracle.dispatch_layout(np.zeros((2, 1), np.int32), np.arange(6), 6, 4)


def test_closed_form_matches_table1_contiguous_rows():
    """Table I's contiguous rows (E=128) agree with the uniform-routing closed
    form within the table's rounding."""
    g = json.load(open(os.path.join(GOLDEN, "table1_contiguous.json")))
    for row in g["rows"]:
        E, k, W = g["E"], row["k"], row["EP"]
        d = expected_distinct_ranks(E, W, k)
        assert abs(d - row["gpus"]) <= 0.03, (row, d)
        assert abs(100 * (1 - d / k) - row["dedup_pct"]) <= 1.0, (row, d)
        assert abs(100 * expected_same_rank_share(E, W, k) - row["same_gpu_pct"]) <= 1.0


@pytest.mark.parametrize("k,W", [(2, 8), (2, 32), (6, 8), (6, 16)])
def test_oracle_dedup_count_matches_closed_form(k, W):
    """With iid logits the oracle's R_d / N is the mean number of distinct ranks
    per token: it must sit within 4 sigma of the closed form."""
    E, N = 128, 4000
    ids = random_ids(N, E, k, seed=k * 100 + W)
    lay = oracle.dispatch_layout(ids, np.arange(E), E, W)
    per_token = lay["rank_member"].sum(axis=1)
    mu = expected_distinct_ranks(E, W, k)
    sigma = per_token.std() / math.sqrt(N)
    assert abs(lay["n_dedup_rows"] / N - mu) <= 4 * sigma + 1e-9
    share = np.mean(per_token == 1)
    p = expected_same_rank_share(E, W, k)
    assert abs(share - p) <= 4 * math.sqrt(max(p * (1 - p), 1e-12) / N) + 1e-9


def test_distinct_ranks_estimate_of_the_phased_section():
    """The pages' estimate W (1 - (1 - 1/W)^k) gives 3.6 at k=8, W=4 (one token);
    drawing experts without replacement (E=64) gives slightly more, and the
    oracle reproduces the exact value."""
    g = json.load(open(os.path.join(GOLDEN, "distinct_ranks_approx.json")))
    W, k = g["W"], g["k"]
    approx = W * (1 - (1 - 1 / W) ** (k * g["m_b"]))
    assert round(approx, 1) == g["approx_ranks_per_token"]
    E, N = 64, 4000
    exact = expected_distinct_ranks(E, W, k)
    assert approx < exact < W
    ids = random_ids(N, E, k, seed=77)
    lay = oracle.dispatch_layout(ids, np.arange(E), E, W)
    per_token = lay["rank_member"].sum(axis=1)
    assert abs(per_token.mean() - exact) <= 4 * per_token.std() / math.sqrt(N)


def test_correlated_placement_reduces_dedup_rows():
    """Co-locating the planted pairs must merge more rows than contiguous
    placement on the same routing ("Expert Coupling" Sec. V-A)."""
    wl = synth.WORKLOADS["correlated_placed"]
    N = 2048
    L = synth.make_logits(wl, N=N)
    ids, _ = oracle.route(L, wl.k)
    contiguous = oracle.dispatch_layout(ids, np.arange(wl.E), wl.E, wl.W)
    placed = oracle.dispatch_layout(ids, synth.make_placement(wl), wl.E, wl.W)
    assert placed["n_dedup_rows"] < contiguous["n_dedup_rows"]
    assert np.array_equal(np.sort(placed["expert_counts"]), np.sort(contiguous["expert_counts"]))
