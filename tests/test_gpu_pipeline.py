"""The microbatch pipeline (two streams, vector-unit stages of one microbatch
overlapping the GEMMs of another) matches the oracle's whole-layer forward
pass within the float tolerance, and returns exactly what the one-shot layer
call returns."""
import numpy as np
import pytest
import torch

import oracle
from cases import SMALL
from combine_warp_top_gb300 import moe, synth
from gpu_util import assert_close, dev_bf16, dev_i32, host_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("name,mb", [("ragged", 128), ("ragged", 77), ("wide", 64), ("e256", 50),
                                     ("odd_h", 150)])
def test_pipeline_is_bit_identical(name, mb, dedup):
    wl = SMALL[name]
    wh = [synth.make_weight(wl, m) for m in ("gate", "up", "down")]
    w = tuple(dev_bf16(a) for a in wh)
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup)
    layer = moe.MoELayer(shape, *w)
    pipe = moe.MicrobatchPipeline(shape, *w, microbatch=mb)
    Lh, xh, rh = synth.make_logits(wl), synth.make_x(wl), synth.make_residual(wl)
    L = torch.from_numpy(Lh).cuda()
    x, res = dev_bf16(xh), dev_bf16(rh)
    want = layer.forward(L, x, res).clone()
    ref = oracle.layer_forward(Lh, xh, *wh, wl.k, wl.W, residual=rh, dedup=dedup)
    for _ in range(2):
        got = pipe.forward(L, x, res)
        torch.cuda.synchronize()
        pipe.check_device_errors()
        assert_close(host_f64(got), ref["out"], f"{name} pipeline out")
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    # the MoE delta alone, against the oracle's
    delta = pipe.forward(L, x, None)
    torch.cuda.synchronize()
    assert_close(host_f64(delta), ref["out"] - oracle.widen_bf16(rh), f"{name} pipeline delta")


def test_pipeline_with_placement_and_shared_expert():
    wl = synth.WORKLOADS["correlated_placed"]
    N = 1000
    w = tuple(dev_bf16(synth.make_weight(wl, m)) for m in ("gate", "up", "down"))
    one = synth.Workload("s", N, wl.H, 1, 1, 256, 1)
    sh = tuple(dev_bf16(synth.make_weight(one, m, seed=5)[0]) for m in ("gate", "up", "down"))
    placement = synth.make_placement(wl)
    pl = dev_i32(placement)
    shape = moe.Shape(N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=True)
    layer = moe.MoELayer(shape, *w, pl, shared=sh)
    pipe = moe.MicrobatchPipeline(shape, *w, pl, microbatch=300, depth=3, shared=sh)
    Lh, xh, rh = synth.make_logits(wl, N=N), synth.make_x(wl, N=N), synth.make_residual(wl, N=N)
    L = torch.from_numpy(Lh).cuda()
    x, res = dev_bf16(xh), dev_bf16(rh)
    want = layer.forward(L, x, res).clone()
    got = pipe.forward(L, x, res)
    torch.cuda.synchronize()
    pipe.check_device_errors()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    # against the oracle: routed experts under the placement, dedup, shared expert
    wh = [synth.make_weight(wl, m) for m in ("gate", "up", "down")]
    shh = tuple(synth.make_weight(one, m, seed=5)[0] for m in ("gate", "up", "down"))
    ref = oracle.layer_forward(Lh, xh, *wh, wl.k, wl.W, placement=placement, residual=rh,
                               dedup=True, shared=shh)
    assert_close(host_f64(got), ref["out"], "pipeline out with placement and shared expert")
