"""moe_dispatch_layout_noalloc, the layout entry point for callers that cannot
allocate device memory at call time (it keeps its scratch in a static device
array instead of a caller workspace).  Its tables must equal those of
moe_dispatch_layout, call after call.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from combine_warp_top_gb300 import moe, synth

pytestmark = pytest.mark.gpu


def _tables(layout):
    return {n: t.cpu().numpy().copy() for n, t in layout.tensors.items()}


def test_noalloc_layout_equals_workspace_layout_twice():
    lib = moe.load()
    wl = synth.WORKLOADS["correlated_placed"]
    N = 3000
    shape = moe.Shape(N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=True)
    L = torch.from_numpy(synth.make_logits(wl, N=N)).cuda()
    ids = torch.empty(N * wl.k, dtype=torch.int32, device="cuda")
    w = torch.empty(N * wl.k, dtype=torch.float32, device="cuda")
    moe.moe_route(L, shape, ids, w)
    placement = torch.from_numpy(synth.make_placement(wl)).cuda()

    ref_layout, ws = moe.Layout(shape), moe.workspace(shape)
    moe.moe_dispatch_layout(ids, placement, shape, ref_layout, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    want = _tables(ref_layout)

    for _ in range(2):  # the static scratch keeps the previous call's contents
        got_layout = moe.Layout(shape)
        st = lib.moe_dispatch_layout_noalloc(
            ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(placement.data_ptr()),
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
