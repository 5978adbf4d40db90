"""Pins of the oracle's correlated-placement search ("Expert Coupling" Sec. V-A
and Appendix A-D, Algorithm 1): co-selection counts, the swap gain, the
balanced best-swap partition and its hierarchical form.  Each is checked
against a direct recomputation of the objective (the within-group total of
co-selection counts), not against the oracle's own formulas."""
import numpy as np
import pytest

import oracle
from combine_warp_top_gb300 import synth


def ids_of(N, E, k, seed):
    return oracle.route(synth.normal_f32(seed, 71, (N, E)), k)[0]


def objective(W, group):
    E = len(group)
    return sum(int(W[a, b]) for a in range(E) for b in range(a + 1, E) if group[a] == group[b])


def swapped(group, a, b):
    g = group.copy()
    g[a], g[b] = group[b], group[a]
    return g


def random_W(E, seed):
    rng = np.random.default_rng(seed)
    M = rng.integers(0, 50, size=(E, E))
    return M + M.T


def test_coselection_is_the_pair_count():
    ids = ids_of(60, 7, 3, 1)
    W = oracle.coselection(ids, 7)
    for a in range(7):
        for b in range(7):
            assert W[a, b] == sum(1 for t in range(60) if a in ids[t] and b in ids[t])
    assert np.array_equal(W, W.T)
    assert np.array_equal(np.diag(W), np.bincount(ids.reshape(-1), minlength=7))
    assert np.triu(W, 1).sum() == 60 * 3 * 2 // 2  # k(k-1)/2 pairs per token


def test_swap_gain_is_the_change_of_the_objective():
    W = random_W(12, 2)
    group = np.arange(12) // 3
    for a in range(12):
        for b in range(a + 1, 12):
            if group[a] != group[b]:
                want = objective(W, swapped(group, a, b)) - objective(W, group)
                assert oracle.swap_gain(W, group, a, b) == want


@pytest.mark.parametrize("E,G,seed", [(8, 2, 3), (12, 3, 4), (12, 4, 5), (16, 4, 6)])
def test_partition_is_balanced_and_locally_optimal(E, G, seed):
    W = random_W(E, seed)
    group, swaps = oracle.partition(W, G, 10_000)
    assert np.array_equal(np.bincount(group, minlength=G), np.full(G, E // G))
    assert objective(W, group) >= objective(W, np.arange(E) // (E // G))
    for a in range(E):  # no improving swap remains
        for b in range(a + 1, E):
            if group[a] != group[b]:
                assert objective(W, swapped(group, a, b)) <= objective(W, group)


def test_each_step_takes_the_best_swap_within_the_budget():
    W = random_W(10, 7)
    group = np.arange(10) // 5
    for budget in range(1, 4):
        best = None
        for a in range(10):
            for b in range(a + 1, 10):
                if group[a] != group[b]:
                    gain = objective(W, swapped(group, a, b)) - objective(W, group)
                    if best is None or gain > best[0]:
                        best = (gain, a, b)
        got, swaps = oracle.partition(W, 2, budget)
        if best[0] <= 0:
            assert np.array_equal(got, group)
            break
        group = swapped(group, best[1], best[2])
        assert swaps == budget and np.array_equal(got, group)


def test_ties_take_the_first_pair_in_lexicographic_order():
    # groups {0,1} {2,3}; the co-selected pairs (0,2) and (1,3) make the swaps
    # (0,3) and (1,2) tie at gain 10; (0,3) comes first
    W = np.zeros((4, 4), np.int64)
    W[0, 2] = W[2, 0] = 5
    W[1, 3] = W[3, 1] = 5
    group, swaps = oracle.partition(W, 2, 1)
    assert group.tolist() == [1, 0, 1, 0] and swaps == 1


def planted_W(E, pairs, noise_seed, strength=100):
    W = random_W(E, noise_seed) // 10
    for a, b in pairs:
        W[a, b] += strength
        W[b, a] += strength
    return W


def test_planted_pairs_are_recovered_on_one_node_and_on_two():
    E = 16
    perm = synth.permutation(0, 72, E)
    pairs = perm.reshape(8, 2)
    W = planted_W(E, pairs, 8)
    for nodes in (1, 2):
        placement, swaps = oracle.correlated_placement(W, 8, nodes=nodes)
        assert sorted(placement.tolist()) == list(range(E))
        rank = np.empty(E, np.int64)
        rank[placement] = np.arange(E) // 2
        for a, b in pairs:
            assert rank[a] == rank[b], (nodes, a, b)
        assert oracle.within_rank_coselection(W, placement, 8) >= 8 * 100


def test_hierarchy_keeps_node_groups():
    """With two nodes, every rank's experts come from the node-level partition."""
    E, ranks = 12, 6
    W = random_W(E, 9)
    node, _ = oracle.partition(W, 2, 10_000)
    placement, _ = oracle.correlated_placement(W, ranks, nodes=2)
    for r in range(ranks):
        members = placement[r * 2:(r + 1) * 2]
        assert set(node[members]) == {r // 3}


def test_searched_placement_merges_more_rows_on_the_correlated_workload():
    """Coupling Sec. V-A: co-locating frequent pairs gives deduplication more
    rows to merge.  The search on the routing's own counts recovers the 20
    planted pairs and beats contiguous placement."""
    wl = synth.WORKLOADS["correlated_contiguous"]
    N = 2048
    ids, _ = oracle.route(synth.make_logits(wl, N=N), wl.k)
    W = oracle.coselection(ids, wl.E)
    placement, swaps = oracle.correlated_placement(W, wl.W)
    rank = np.empty(wl.E, np.int64)
    rank[placement] = np.arange(wl.E) // (wl.E // wl.W)
    for a, b in synth.hot_pairs(wl):
        assert rank[a] == rank[b]
    searched = oracle.dispatch_layout(ids, placement, wl.E, wl.W)["n_dedup_rows"]
    contiguous = oracle.dispatch_layout(ids, np.arange(wl.E), wl.E, wl.W)["n_dedup_rows"]
    planted = oracle.dispatch_layout(ids, synth.make_placement(synth.WORKLOADS["correlated_placed"]),
                                     wl.E, wl.W)["n_dedup_rows"]
    assert searched < contiguous
    assert searched <= planted
