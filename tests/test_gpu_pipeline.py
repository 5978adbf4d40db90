"""The microbatch pipeline (two streams, vector-unit stages of one microbatch
overlapping the GEMMs of another) returns exactly what the one-shot layer call
returns."""
import numpy as np
import pytest
import torch

from cases import SMALL
from combine_warp_top_gb300 import moe, synth
from gpu_util import dev_bf16, dev_i32

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("name,mb", [("ragged", 128), ("ragged", 77), ("wide", 64), ("e256", 50),
                                     ("odd_h", 150)])
def test_pipeline_is_bit_identical(name, mb, dedup):
    wl = SMALL[name]
    w = tuple(dev_bf16(synth.make_weight(wl, m)) for m in ("gate", "up", "down"))
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup)
    layer = moe.MoELayer(shape, *w)
    pipe = moe.MicrobatchPipeline(shape, *w, microbatch=mb)
    L = torch.from_numpy(synth.make_logits(wl)).cuda()
    x, res = dev_bf16(synth.make_x(wl)), dev_bf16(synth.make_residual(wl))
    want = layer.forward(L, x, res).clone()
    for _ in range(2):
        got = pipe.forward(L, x, res)
        torch.cuda.synchronize()
        pipe.check_device_errors()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_pipeline_with_placement_and_shared_expert():
    wl = synth.WORKLOADS["correlated_placed"]
    N = 1000
    w = tuple(dev_bf16(synth.make_weight(wl, m)) for m in ("gate", "up", "down"))
    one = synth.Workload("s", N, wl.H, 1, 1, 256, 1)
    sh = tuple(dev_bf16(synth.make_weight(one, m, seed=5)[0]) for m in ("gate", "up", "down"))
    pl = dev_i32(synth.make_placement(wl))
    shape = moe.Shape(N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=True)
    layer = moe.MoELayer(shape, *w, pl, shared=sh)
    pipe = moe.MicrobatchPipeline(shape, *w, pl, microbatch=300, depth=3, shared=sh)
    L = torch.from_numpy(synth.make_logits(wl, N=N)).cuda()
    x, res = dev_bf16(synth.make_x(wl, N=N)), dev_bf16(synth.make_residual(wl, N=N))
    want = layer.forward(L, x, res).clone()
    got = pipe.forward(L, x, res)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
