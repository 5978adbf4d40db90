"""The library's host-side placement search (moe_placement_search, C++) against
the oracle's restatement of Algorithm 1 ("Expert Coupling" Appendix A-D):
identical placements, bit for bit.  Runs on the CPU: the search is host code."""
import numpy as np
import pytest
import torch

import oracle
from combine_warp_top_gb300 import build as libbuild
from combine_warp_top_gb300 import moe, synth


@pytest.fixture(scope="module", autouse=True)
def lib():
    libbuild.build()
    return moe.load()


def random_W(E, seed, hi=50):
    rng = np.random.default_rng(seed)
    M = rng.integers(0, hi, size=(E, E))
    return (M + M.T).astype(np.int32)


@pytest.mark.parametrize("E,ranks,nodes,seed", [(8, 4, 1, 1), (12, 3, 1, 2), (16, 8, 2, 3),
                                                (24, 6, 3, 4), (32, 8, 1, 5), (64, 32, 1, 6),
                                                (64, 16, 4, 7)])
def test_search_equals_oracle(E, ranks, nodes, seed):
    W = random_W(E, seed)
    got, swaps = moe.moe_placement_search(torch.from_numpy(W), ranks, nodes)
    want, want_swaps = oracle.correlated_placement(W, ranks, nodes)
    assert np.array_equal(got.numpy(), want)
    assert swaps == want_swaps


def test_search_budget_and_ties():
    W = np.zeros((4, 4), np.int32)
    W[0, 2] = W[2, 0] = 5
    W[1, 3] = W[3, 1] = 5
    got, swaps = moe.moe_placement_search(torch.from_numpy(W), 2, 1, max_swaps=1)
    want, _ = oracle.correlated_placement(W, 2, 1, max_swaps=1)
    assert np.array_equal(got.numpy(), want) and swaps == 1
    got0, swaps0 = moe.moe_placement_search(torch.from_numpy(W), 2, 1, max_swaps=0)
    assert got0.tolist() == [0, 1, 2, 3] and swaps0 == 0


def test_search_on_the_correlated_workload_counts():
    wl = synth.WORKLOADS["correlated_contiguous"]
    ids, _ = oracle.route(synth.make_logits(wl, N=2048), wl.k)
    W = oracle.coselection(ids, wl.E).astype(np.int32)
    got, _ = moe.moe_placement_search(torch.from_numpy(W), wl.W)
    want, _ = oracle.correlated_placement(W, wl.W)
    assert np.array_equal(got.numpy(), want)


def test_large_search_is_balanced_and_locally_optimal():
    E, ranks = 256, 8
    W = random_W(E, 11, hi=1000)
    got, swaps = moe.moe_placement_search(torch.from_numpy(W), ranks)
    p = got.numpy()
    assert sorted(p.tolist()) == list(range(E))
    group = np.empty(E, np.int64)
    group[p] = np.arange(E) // (E // ranks)
    Wl = W.astype(np.int64)
    onehot = np.eye(ranks, dtype=np.int64)[group]
    conn = Wl @ onehot - np.diag(Wl)[:, None] * onehot      # excludes the expert itself
    ga = group[:, None]
    gb = group[None, :]
    gain = (conn[np.arange(E)[:, None], gb] - conn[np.arange(E), group][:, None]
            + conn[np.arange(E)[None, :], ga] - conn[np.arange(E), group][None, :] - 2 * Wl)
    gain[ga == gb] = 0
    assert gain.max() <= 0


def test_search_rejects_bad_arguments(lib):
    W = torch.zeros(12, 12, dtype=torch.int32)
    with pytest.raises(moe.MoeError):
        moe.moe_placement_search(W, 5)        # 5 does not divide 12
    with pytest.raises(moe.MoeError):
        moe.moe_placement_search(W, 6, 4)     # 4 does not divide 6
