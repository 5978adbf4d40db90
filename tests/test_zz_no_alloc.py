"""moe_dispatch_layout_noalloc, the layout entry point for callers that cannot
allocate device memory at call time (it keeps its scratch in a static device
array instead of a caller workspace).  Its tables must equal those of
moe_dispatch_layout, call after call.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from combine_warp_top_gb300 import moe, synth

pytestmark = pytest.mark.gpu


def _tables(layout):
    return {n: t.cpu().numpy().copy() for n, t in layout.tensors.items()}


# N = 300 and 3000: two and twelve count blocks, whose tables the scatter
# blocks scan themselves; N = 70000: 274 blocks, whose 70 KB (plain) and
# 105 KB (dedup) tables take the separate scan launch.  Plain and dedup;
# contiguous placement (NULL) and the correlated workload's permutation.
@pytest.mark.parametrize("N", [300, 3000, 70000])
@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("placed", [False, True])
def test_noalloc_layout_equals_workspace_layout_twice(N, dedup, placed):
    lib = moe.load()
    wl = synth.WORKLOADS["correlated_placed"]
    shape = moe.Shape(N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup)
    L = torch.from_numpy(synth.make_logits(wl, N=N)).cuda()
    ids = torch.empty(N * wl.k, dtype=torch.int32, device="cuda")
    w = torch.empty(N * wl.k, dtype=torch.float32, device="cuda")
    moe.moe_route(L, shape, ids, w)
    placement_h = synth.make_placement(wl) if placed else np.arange(wl.E, dtype=np.int32)
    placement = torch.from_numpy(placement_h).cuda() if placed else None

    ref_layout, ws = moe.Layout(shape), moe.workspace(shape)
    moe.moe_dispatch_layout(ids, placement, shape, ref_layout, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    want = _tables(ref_layout)
    # the workspace form is itself the oracle's layout
    ref = oracle.dispatch_layout(ids.view(N, wl.k).cpu().numpy(), placement_h, wl.E, wl.W)
    for key in ("expert_counts", "expert_offsets", "rank_offsets", "row_token"):
        assert np.array_equal(want[key][:len(ref[key])], ref[key]), key
    assert np.array_equal(want["pair_row"].reshape(N, wl.k), ref["pair_row"])
    if dedup:
        Rd = ref["n_dedup_rows"]
        assert int(want["n_dedup_rows"][0]) == Rd
        assert np.array_equal(want["dedup_row_token"][:Rd], ref["dedup_row_token"])
        assert np.array_equal(want["pair_dedup_row"].reshape(N, wl.k), ref["pair_dedup_row"])

    for _ in range(2):  # the static scratch keeps the previous call's contents
        got_layout = moe.Layout(shape)
        st = lib.moe_dispatch_layout_noalloc(
            ctypes.c_void_p(ids.data_ptr()),
            None if placement is None else ctypes.c_void_p(placement.data_ptr()),
            ctypes.byref(shape.c()), ctypes.byref(got_layout.c),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, moe.moe_status_str(st)
        torch.cuda.synchronize()
        got = _tables(got_layout)
        for name in want:  # integer tables: the tolerance is exact equality
            assert np.array_equal(got[name], want[name]), name


def test_noalloc_rejects_shapes_beyond_its_static_scratch():
    lib = moe.load()
    big = moe.Shape(1 << 20, 8, 1024, 2, 1024, 8)  # per-block counts alone exceed 1 MiB
    assert moe.moe_workspace_bytes(big) > (1 << 20)
    lay = moe.Layout(moe.Shape(1, 8, 1024, 2, 1024, 8))  # never touched: rejected first
    st = lib.moe_dispatch_layout_noalloc(None, None, ctypes.byref(big.c()), ctypes.byref(lay.c),
                                         None)
    assert st == 3  # MOE_ERR_WORKSPACE
