"""Edge cases of the CUDA path against the oracle: the largest expert count
(the layout kernels' large shared-memory configuration), one expert, one
token, and widths below one TMA box."""
import numpy as np
import pytest
import torch

import oracle
from combine_warp_top_gb300 import moe, synth
from gpu_util import assert_close, dev_bf16, dev_i32, host_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,E,k,W", [(3000, 1024, 32, 1024), (2000, 1024, 8, 4),
                                     (700, 512, 16, 512), (5, 1024, 3, 256)])
def test_layout_largest_expert_counts(N, E, k, W):
    L = synth.normal_f32(0, 91, (N, E))
    ids, _ = oracle.route(L, k)
    shape = moe.Shape(N, 8, E, k, W, 8, dedup=True)
    lay = moe.Layout(shape)
    ws = moe.workspace(shape)
    moe.moe_dispatch_layout(dev_i32(ids), None, shape, lay, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    ref = oracle.dispatch_layout(ids, np.arange(E), E, W)
    got = {n: t.cpu().numpy() for n, t in lay.tensors.items()}
    for key in ("expert_counts", "expert_offsets", "rank_offsets", "row_token", "dedup_counts",
                "dedup_offsets", "expand_src"):
        assert np.array_equal(got[key][:len(ref[key])], ref[key]), key
    assert np.array_equal(got["pair_row"].reshape(N, k), ref["pair_row"])
    assert np.array_equal(got["pair_dedup_row"].reshape(N, k), ref["pair_dedup_row"])
    assert int(got["n_dedup_rows"][0]) == ref["n_dedup_rows"]


def run_layer(wl, dedup=False, gemm="auto"):
    w = [synth.make_weight(wl, m) for m in ("gate", "up", "down")]
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup, gemm=gemm)
    layer = moe.MoELayer(shape, *[dev_bf16(a) for a in w])
    L, x, res = synth.make_logits(wl), synth.make_x(wl), synth.make_residual(wl)
    out = layer.forward(torch.from_numpy(L).cuda(), dev_bf16(x), dev_bf16(res))
    torch.cuda.synchronize()
    layer.check_device_errors()
    ref = oracle.layer_forward(L, x, *w, wl.k, wl.W, residual=res, dedup=dedup)
    assert np.array_equal(layer.topk_ids.view(wl.N, wl.k).cpu().numpy(), ref["topk_ids"])
    assert_close(host_f64(layer.y[:wl.N * wl.k]), ref["y"], "y")
    assert_close(host_f64(out), ref["out"], "out")


EDGE = [
    synth.Workload("one_expert", 300, 128, 1, 1, 128, 1),
    synth.Workload("one_token", 1, 256, 8, 2, 128, 2),
    synth.Workload("one_token_one_expert", 1, 64, 1, 1, 64, 1),
    synth.Workload("narrow16", 200, 16, 4, 2, 16, 2),
    synth.Workload("narrow8", 130, 8, 4, 2, 8, 4),
    synth.Workload("wide_i_small_h", 300, 64, 4, 2, 1000, 2),
]


@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("wl", EDGE, ids=lambda w: w.name)
def test_layer_edge_shapes(wl, dedup):
    run_layer(wl, dedup)


@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("wl", EDGE, ids=lambda w: w.name)
def test_layer_edge_shapes_on_cta_pairs(wl, dedup):
    """The same shapes on the CTA-pair GEMMs (named in the shape): fewer tiles
    than pairs, so most pairs find the tile queue exhausted at once; tiles of
    one row."""
    run_layer(wl, dedup, gemm="pair")


def test_misaligned_view_is_refused_and_the_context_survives():
    """A contiguous bf16 view that starts one element into its buffer is off the
    16-byte grid the kernels' vector loads need: the call is refused on the host
    with an invalid-argument status, nothing is launched, and the same call on
    an aligned copy then matches the oracle."""
    wl = synth.Workload("align", 64, 128, 8, 2, 64, 2)
    ids, w64 = oracle.route(synth.make_logits(wl), wl.k)
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I)
    lay = moe.Layout(shape)
    ws = moe.workspace(shape)
    moe.moe_dispatch_layout(dev_i32(ids), None, shape, lay, ws)
    ref = oracle.dispatch_layout(ids, np.arange(wl.E), wl.E, wl.W)
    y = synth.normal_bf16(0, 65, (shape.R, wl.H))
    res = synth.make_residual(wl)
    w32 = torch.from_numpy(w64.astype(np.float32)).cuda()
    buf = torch.empty(shape.R * wl.H + 8, dtype=torch.bfloat16, device="cuda")
    y_odd = buf[1:1 + shape.R * wl.H].view(shape.R, wl.H)
    y_odd.copy_(dev_bf16(y))
    out = torch.empty(wl.N, wl.H, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as info:
        moe.moe_combine(y_odd, w32, lay, shape, None, dev_bf16(res), out)
    assert info.value.status == 1  # MOE_ERR_INVALID_ARG
    assert moe.moe_get_error(ws) == 0
    moe.moe_combine(y_odd.clone(), w32, lay, shape, None, dev_bf16(res), out)
    torch.cuda.synchronize()
    want = oracle.combine(oracle.widen_bf16(y), w64.astype(np.float32).astype(np.float64),
                          ref["pair_row"], res)
    assert_close(host_f64(out), want, "combine after a refused call")
