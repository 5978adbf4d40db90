"""End-to-end parity of moe_layer_forward (one call through the C ABI) against
the oracle, with and without dedup and residual, and the C ABI's error paths."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from cases import SMALL
from combine_warp_top_gb300 import moe, synth
from gpu_util import assert_close, dev_bf16, dev_i32, host_f64, host_u16

pytestmark = pytest.mark.gpu


def build_layer(wl, dedup, placement=None, N=None, gemm="auto"):
    N = wl.N if N is None else N
    wg, wu, wd = (synth.make_weight(wl, w) for w in ("gate", "up", "down"))
    shape = moe.Shape(N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup, gemm=gemm)
    layer = moe.MoELayer(shape, dev_bf16(wg), dev_bf16(wu), dev_bf16(wd),
                         None if placement is None else dev_i32(placement))
    return layer, (wg, wu, wd)


def check_layer(wl, dedup, placement=None, N=None):
    N = wl.N if N is None else N
    layer, (wg, wu, wd) = build_layer(wl, dedup, placement, N)
    L = synth.make_logits(wl, N=N)
    x, res = synth.make_x(wl, N=N), synth.make_residual(wl, N=N)
    out = layer.forward(torch.from_numpy(L).cuda(), dev_bf16(x), dev_bf16(res))
    torch.cuda.synchronize()
    layer.check_device_errors()
    got = host_f64(out)
    ids = layer.topk_ids.view(N, wl.k).cpu().numpy()
    ref = oracle.layer_forward(L, x, wg, wu, wd, wl.k, wl.W, placement=placement, residual=res,
                               dedup=dedup)
    assert np.array_equal(ids, ref["topk_ids"])
    assert np.array_equal(layer.layout["expert_counts"].cpu().numpy(),
                          ref["layout"]["expert_counts"])
    if dedup:
        assert int(layer.layout["n_dedup_rows"].item()) == ref["layout"]["n_dedup_rows"]
    assert_close(got, ref["out"], "out")
    # the MoE delta alone: residual NULL
    out2 = layer.forward(torch.from_numpy(L).cuda(), dev_bf16(x), None)
    torch.cuda.synchronize()
    delta = ref["out"] - oracle.widen_bf16(res)
    assert_close(host_f64(out2), delta, "MoE delta")


@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("name", list(SMALL))
def test_layer_small(name, dedup):
    check_layer(SMALL[name], dedup)


@pytest.mark.parametrize("name", ["correlated_contiguous", "correlated_placed"])
def test_layer_correlated_reduced(name):
    wl = synth.WORKLOADS[name]
    check_layer(wl, True, synth.make_placement(wl), N=512)


def test_layer_skewed_reduced():
    wl = synth.WORKLOADS["skewed"]
    small = synth.Workload("skewed_small", 1024, 256, wl.E, wl.k, 256, wl.W, logits="zipf",
                           zipf_alpha=1.2)
    check_layer(small, False)


def test_layer_empty_batch_is_noop():
    wl = SMALL["tiny"]
    layer, _ = build_layer(wl, False, N=0)
    empty = torch.empty(0, wl.E, dtype=torch.float32, device="cuda")
    layer.forward(empty, torch.empty(0, wl.H, dtype=torch.bfloat16, device="cuda"), None)
    torch.cuda.synchronize()
    layer.check_device_errors()


def test_repeated_calls_are_bitwise_stable():
    wl = SMALL["ragged"]
    layer, _ = build_layer(wl, True)
    L = torch.from_numpy(synth.make_logits(wl)).cuda()
    x, res = dev_bf16(synth.make_x(wl)), dev_bf16(synth.make_residual(wl))
    first = layer.forward(L, x, res).clone()
    for _ in range(3):
        again = layer.forward(L, x, res)
        torch.cuda.synchronize()
        assert torch.equal(first.view(torch.int16), again.view(torch.int16))


# ---- error paths: checked on the host, nothing launched ---------------------------------

def test_invalid_arguments_are_rejected():
    lib = moe.load()
    wl = SMALL["tiny"]
    good = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I)
    assert moe.moe_workspace_bytes(good) > 0
    for bad in (moe.Shape(64, 128, 8, 9, 2, 256), moe.Shape(64, 128, 8, 2, 3, 256),
                moe.Shape(-1, 128, 8, 2, 2, 256), moe.Shape(64, 128, 8, 0, 2, 256)):
        assert moe.moe_workspace_bytes(bad) == 0
    assert lib.moe_workspace_bytes(moe.MoeShape(64, 130, 8, 2, 2, 256)) == 0  # H % 8
    assert lib.moe_workspace_bytes(moe.MoeShape(64, 128, 2048, 2, 2, 256)) == 0  # E too large
    ids = torch.zeros(wl.N * wl.k, dtype=torch.int32, device="cuda")
    w = torch.zeros(wl.N * wl.k, dtype=torch.float32, device="cuda")
    st = lib.moe_route(None, ctypes.byref(good.c()), ids.data_ptr(), w.data_ptr(), None)
    assert st == 1
    lay = moe.Layout(good)
    small_ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_dispatch_layout(ids, None, good, lay, small_ws)
    assert e.value.status == 3
    dshape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, True)
    ws = moe.workspace(dshape)
    # a plain layout has no dedup arrays: the binding refuses it for a dedup
    # shape, and so does the C call it would make
    with pytest.raises(ValueError, match="another shape"):
        moe.moe_dispatch_layout(ids, None, dshape, lay, ws)
    st = lib.moe_dispatch_layout(ids.data_ptr(), None, ctypes.byref(dshape.c()),
                                 ctypes.byref(lay.c), ws.data_ptr(), ws.numel(), None)
    assert st == 1


def test_bad_placement_is_reported_by_the_device():
    """A placement that is not a permutation is flagged in the workspace error
    word; the kernels stay in bounds."""
    wl = SMALL["tiny"]
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=True)
    ids, _ = oracle.route(synth.make_logits(wl), wl.k)
    lay = moe.Layout(shape)
    ws = moe.workspace(shape)
    bad = np.arange(wl.E, dtype=np.int32)
    bad[3] = 2
    moe.moe_dispatch_layout(dev_i32(ids), dev_i32(bad), shape, lay, ws)
    assert moe.moe_get_error(ws) == 1
    assert moe.moe_get_error(ws) == 0  # cleared by the read
    moe.moe_dispatch_layout(dev_i32(ids), None, shape, lay, ws)
    assert moe.moe_get_error(ws) == 0


@pytest.mark.parametrize("graphs", [True, False])
def test_host_pipeline_matches_device_forward(graphs):
    """The overlapped host-buffer path returns, batch by batch, exactly what the
    device-resident call returns, whether it replays a captured graph per
    buffer set or calls the layer directly."""
    wl = SMALL["wide"]
    layer, _ = build_layer(wl, False)
    batches, want = [], []
    for seed in range(4):
        L = torch.from_numpy(synth.make_logits(wl, seed)).pin_memory()
        x = torch.from_numpy(synth.make_x(wl, seed).view(np.int16)).view(torch.bfloat16).pin_memory()
        r = torch.from_numpy(synth.make_residual(wl, seed).view(np.int16)).view(torch.bfloat16).pin_memory()
        out = torch.empty(wl.N, wl.H, dtype=torch.bfloat16).pin_memory()
        batches.append((L, x, r, out))
        want.append(layer.forward(L.cuda(), x.cuda(), r.cuda()).cpu().clone())
    pipe = moe.HostPipeline(layer, graphs=graphs)
    assert (pipe.graphs is not None) == graphs
    pipe.run(batches)
    torch.cuda.synchronize()
    for (_, _, _, out), w in zip(batches, want):
        assert torch.equal(out.view(torch.int16), w.view(torch.int16))


def test_wait_timeout_is_reported_and_the_context_survives():
    """A device-side wait on a barrier that nothing completes gives up after its
    limit (about 1 ms of SM clock here), records MOE_ERR_TIMEOUT, and the next
    layer call runs normally."""
    wl = SMALL["tiny"]
    layer, _ = build_layer(wl, False)
    moe.moe_selftest_wait_timeout(layer.ws, 2_000_000)
    assert moe.moe_get_error(layer.ws) == 5  # MOE_ERR_TIMEOUT
    assert moe.moe_get_error(layer.ws) == 0
    L = torch.from_numpy(synth.make_logits(wl)).cuda()
    x, res = dev_bf16(synth.make_x(wl)), dev_bf16(synth.make_residual(wl))
    a = layer.forward(L, x, res).clone()
    torch.cuda.synchronize()
    layer.check_device_errors()
    b = layer.forward(L, x, res)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("dedup", [False, True])
def test_cuda_graph_replay_matches_eager(dedup):
    """The whole layer captured once as a CUDA graph and replayed on new
    contents of the same input buffers gives the eager results bit for bit."""
    wl = SMALL["ragged"]
    layer, _ = build_layer(wl, dedup)
    L = torch.from_numpy(synth.make_logits(wl, 0)).cuda()
    x, res = dev_bf16(synth.make_x(wl, 0)), dev_bf16(synth.make_residual(wl, 0))
    g = layer.capture(L, x, res)
    for seed in (1, 2):
        L.copy_(torch.from_numpy(synth.make_logits(wl, seed)))
        x.copy_(dev_bf16(synth.make_x(wl, seed)))
        res.copy_(dev_bf16(synth.make_residual(wl, seed)))
        g.replay()
        torch.cuda.synchronize()
        got = layer.out.clone()
        want = layer.forward(L, x, res)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    layer.check_device_errors()


def test_fused_dispatch_and_staged_forms_agree():
    """On a shape whose plain dispatch is fused into the gate/up GEMM (the
    single-CTA kernel, named in the shape), the layer gives bit for bit the
    output of the staged form (dispatch copy, then the CTA-pair GEMMs, named
    in the shape); which form runs follows from the shape alone."""
    wl = SMALL["wide"]
    fused_layer, _ = build_layer(wl, False, gemm="single")
    assert fused_layer.fused_dispatch and moe.moe_layer_skips_dispatch(fused_layer.shape)
    assert fused_layer.xd.shape[0] == 1
    layer, _ = build_layer(wl, False, gemm="pair")
    assert not layer.fused_dispatch and not moe.moe_layer_skips_dispatch(layer.shape)
    assert layer.xd.shape[0] == layer.shape.R
    L = torch.from_numpy(synth.make_logits(wl)).cuda()
    x, res = dev_bf16(synth.make_x(wl)), dev_bf16(synth.make_residual(wl))
    fused = fused_layer.forward(L, x, res).clone()
    staged = layer.forward(L, x, res).clone()
    torch.cuda.synchronize()
    fused_layer.check_device_errors()
    layer.check_device_errors()
    # same K order in both GEMM kernels and the same combine: identical bits
    assert torch.equal(fused.view(torch.int16), staged.view(torch.int16))
    # and the dispatched rows the staged form wrote are the oracle's
    ref = oracle.dispatch_layout(layer.topk_ids.view(wl.N, wl.k).cpu().numpy(),
                                 np.arange(wl.E), wl.E, wl.W)
    assert np.array_equal(host_u16(layer.xd), oracle.dispatch(synth.make_x(wl), ref["row_token"]))


@pytest.mark.parametrize("name,N,gemm", [("correlated_placed", 4096, "pair"),
                                         ("mixtral", 2048, "pair"),
                                         ("skewed", 4096, "auto")])
def test_layer_is_bit_identical_run_to_run(name, N, gemm):
    """Ten forwards of the same inputs give the same bits in every output: the
    CTA-pair GEMM hands tiles out dynamically and the plain combine runs on
    persistent warps, so which SM computes what changes from run to run, but
    no sum depends on it (each tile's K order and each token's j order are
    fixed)."""
    wl = synth.WORKLOADS[name]
    w = [dev_bf16(synth.make_weight(wl, m)) for m in ("gate", "up", "down")]
    pl = None if wl.placement == "contiguous" else dev_i32(synth.make_placement(wl))
    shape = moe.Shape(N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=wl.dedup, gemm=gemm)
    layer = moe.MoELayer(shape, *w, pl)
    L = torch.from_numpy(synth.make_logits(wl, N=N)).cuda()
    x, res = dev_bf16(synth.make_x(wl, N=N)), dev_bf16(synth.make_residual(wl, N=N))
    first = None
    for _ in range(10):
        out = layer.forward(L, x, res)
        torch.cuda.synchronize()
        got = [t.clone() for t in (out, layer.h, layer.y, layer.topk_w)] + \
              [t.clone() for t in layer.layout.tensors.values()]
        if first is None:
            first = got
        else:
            for a, b in zip(first, got):
                assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    layer.check_device_errors()
