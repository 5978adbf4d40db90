"""Co-selection counts on the GPU (moe_coselection) against the oracle, and
the whole correlated-placement path ("Expert Coupling" Sec. V-A): counts on the
GPU, search on the host, dispatch layout under the found placement."""
import numpy as np
import pytest
import torch

import oracle
from combine_warp_top_gb300 import moe, synth
from gpu_util import dev_i32

pytestmark = pytest.mark.gpu


def gpu_coselection(ids, shape):
    W = torch.full((shape.E, shape.E), -7, dtype=torch.int32, device="cuda")  # overwritten
    ws = moe.workspace(shape)
    moe.moe_coselection(dev_i32(ids), shape, W, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    return W.cpu().numpy()


@pytest.mark.parametrize("N,E,k", [(1, 8, 2), (300, 8, 2), (1000, 64, 6), (777, 128, 8),
                                   (500, 256, 8), (64, 1024, 32)])
def test_coselection_bit_exact(N, E, k):
    ids, _ = oracle.route(synth.normal_f32(3, 81, (N, E)), k)
    shape = moe.Shape(N, 8, E, k, 1, 8)
    assert np.array_equal(gpu_coselection(ids, shape), oracle.coselection(ids, E))


@pytest.mark.parametrize("name", ["correlated_contiguous", "skewed", "deepseek_v3"])
def test_coselection_full_size(name):
    wl = synth.WORKLOADS[name]
    ids, _ = oracle.route(synth.make_logits(wl), wl.k)
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I)
    assert np.array_equal(gpu_coselection(ids, shape), oracle.coselection(ids, wl.E))


def test_searched_placement_end_to_end():
    """On the full correlated workload: the search recovers the 20 planted pairs,
    and the layout under the found placement is bit-exact to the oracle's, with
    fewer dedup rows than contiguous placement."""
    wl = synth.WORKLOADS["correlated_contiguous"]
    L = torch.from_numpy(synth.make_logits(wl)).cuda()
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=True)
    ids = torch.empty(wl.N * wl.k, dtype=torch.int32, device="cuda")
    w = torch.empty(wl.N * wl.k, dtype=torch.float32, device="cuda")
    moe.moe_route(L, shape, ids, w)
    ws = moe.workspace(shape)
    W = torch.empty(wl.E, wl.E, dtype=torch.int32, device="cuda")
    moe.moe_coselection(ids, shape, W, ws)
    placement, swaps = moe.moe_placement_search(W.cpu(), wl.W)
    assert swaps > 0
    rank = np.empty(wl.E, np.int64)
    rank[placement.numpy()] = np.arange(wl.E) // (wl.E // wl.W)
    for a, b in synth.hot_pairs(wl):
        assert rank[a] == rank[b]
    lay = moe.Layout(shape)
    moe.moe_dispatch_layout(ids, placement.cuda(), shape, lay, ws)
    torch.cuda.synchronize()
    ids_h = ids.view(wl.N, wl.k).cpu().numpy()
    ref = oracle.dispatch_layout(ids_h, placement.numpy(), wl.E, wl.W)
    assert int(lay["n_dedup_rows"].item()) == ref["n_dedup_rows"]
    assert np.array_equal(lay["pair_dedup_row"].view(wl.N, wl.k).cpu().numpy(), ref["pair_dedup_row"])
    contiguous = oracle.dispatch_layout(ids_h, np.arange(wl.E), wl.E, wl.W)["n_dedup_rows"]
    assert ref["n_dedup_rows"] < contiguous
