"""GPU parity of the widened rows: the full-softmax router variant and the
shared expert (dense SwiGLU over every token, added in the combine)."""
import numpy as np
import pytest
import torch

import oracle
from cases import SMALL
from combine_warp_top_gb300 import moe, synth
from gpu_util import assert_close, dev_bf16, host_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "wide", "e256", "k_eq_e"])
def test_route_full_softmax(name):
    wl = SMALL[name]
    L = synth.make_logits(wl)
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I)
    ids = torch.empty(wl.N * wl.k, dtype=torch.int32, device="cuda")
    w = torch.empty(wl.N * wl.k, dtype=torch.float32, device="cuda")
    moe.moe_route_full_softmax(torch.from_numpy(L).cuda(), shape, ids, w)
    torch.cuda.synchronize()
    ref_ids, ref_w = oracle.route(L, wl.k, renormalize=False)
    assert np.array_equal(ids.view(wl.N, wl.k).cpu().numpy(), ref_ids)
    np.testing.assert_allclose(w.view(wl.N, wl.k).cpu().numpy(), ref_w, rtol=0, atol=2e-6)


def shared_weights(wl, I_s, seed=0):
    one = synth.Workload("shared", wl.N, wl.H, 1, 1, I_s, 1)
    return tuple(synth.make_weight(one, m, seed=seed + 100)[0] for m in ("gate", "up", "down"))


@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("name,I_s", [("tiny", 256), ("ragged", 200), ("odd_h", 136),
                                      ("wide", 384)])
def test_layer_with_shared_expert(name, I_s, dedup):
    wl = SMALL[name]
    wg, wu, wd = (synth.make_weight(wl, m) for m in ("gate", "up", "down"))
    sh = shared_weights(wl, I_s)
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup)
    layer = moe.MoELayer(shape, dev_bf16(wg), dev_bf16(wu), dev_bf16(wd),
                         shared=tuple(dev_bf16(m) for m in sh))
    L, x, res = synth.make_logits(wl), synth.make_x(wl), synth.make_residual(wl)
    out = layer.forward(torch.from_numpy(L).cuda(), dev_bf16(x), dev_bf16(res))
    torch.cuda.synchronize()
    layer.check_device_errors()
    ref = oracle.layer_forward(L, x, wg, wu, wd, wl.k, wl.W, residual=res, dedup=dedup, shared=sh)
    assert_close(host_f64(layer.h_s), ref["h_shared"], "shared h")
    assert_close(host_f64(layer.y_s), ref["y_shared"], "shared y")
    assert_close(host_f64(out), ref["out"], "out")
    delta = layer.forward(torch.from_numpy(L).cuda(), dev_bf16(x), None)
    torch.cuda.synchronize()
    assert_close(host_f64(delta), ref["out"] - oracle.widen_bf16(res), "MoE delta")


def test_shared_expert_full_size_deepseek():
    """DeepSeek-V3 shape with its one shared expert (width 2048), sampled tokens."""
    wl = synth.WORKLOADS["deepseek_v3"]
    I_s = 2048
    one = synth.Workload("shared", wl.N, wl.H, 1, 1, I_s, 1)
    sh_d = []
    for m, stream in (("gate", 103), ("up", 104), ("down", 105)):
        rows, cols = (I_s, wl.H) if m != "down" else (wl.H, I_s)
        t = torch.empty(rows, cols, dtype=torch.bfloat16, device="cuda")
        sh_d.append(synth.normal_bf16_device(t, 0, stream, std=0.02))
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I)
    layer = moe.MoELayer(shape, synth.make_weight_device(wl, "gate"),
                         synth.make_weight_device(wl, "up"), synth.make_weight_device(wl, "down"),
                         shared=tuple(sh_d))
    L, x, res = synth.make_logits(wl), synth.make_x(wl), synth.make_residual(wl)
    out = layer.forward(torch.from_numpy(L).cuda(),
                        torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda(),
                        torch.from_numpy(res.view(np.int16)).view(torch.bfloat16).cuda())
    torch.cuda.synchronize()
    layer.check_device_errors()
    toks = np.array([0, 1234, 4095])
    ids, w = oracle.route(L, wl.k)
    sh_h = tuple(synth.normal_bf16(0, s, shp, std=0.02) for s, shp in
                 ((103, (I_s, wl.H)), (104, (I_s, wl.H)), (105, (wl.H, I_s))))

    def weights_of(e):
        return tuple(synth.make_weight(wl, m, experts=[e])[0] for m in ("gate", "up", "down"))

    routed, _ = oracle.token_outputs(x[toks], ids[toks], w[toks], weights_of, res[toks])
    _, y_s = oracle.shared_expert(x[toks], sh_h)
    assert_close(host_f64(out[torch.from_numpy(toks).cuda()]), routed + y_s, "out with shared")


@pytest.mark.parametrize("N,E,k", [(64, 8, 2), (1000, 64, 6), (4096, 256, 8), (500, 1024, 32),
                                   (300, 7, 7)])
def test_route_sigmoid_bias(N, E, k):
    L = synth.normal_f32(0, 93, (N, E))
    b = synth.normal_f32(0, 94, (E,), std=0.05)
    shape = moe.Shape(N, 8, E, k, 1, 8)
    ids = torch.empty(N * k, dtype=torch.int32, device="cuda")
    w = torch.empty(N * k, dtype=torch.float32, device="cuda")
    moe.moe_route_sigmoid_bias(torch.from_numpy(L).cuda(), torch.from_numpy(b).cuda(), shape, ids, w)
    torch.cuda.synchronize()
    ref_ids, ref_w = oracle.route_sigmoid_bias(L, b, k)
    assert np.array_equal(ids.view(N, k).cpu().numpy(), ref_ids)
    np.testing.assert_allclose(w.view(N, k).cpu().numpy(), ref_w, rtol=0, atol=2e-6)
