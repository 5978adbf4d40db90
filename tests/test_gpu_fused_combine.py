"""The combine fused into the down GEMM's epilogue (moe_ffn_down_combine): each
expert output row, scaled by its routing weight, is added into an fp32
accumulator by atomics, then the residual is added and the sum rounded to bf16.
Checked against the oracle (within the float tolerance; the atomics fix no
order) and against the unfused layer."""
import numpy as np
import pytest
import torch

import oracle
from cases import SMALL
from combine_warp_top_gb300 import moe, synth
from gpu_util import assert_close, dev_bf16, host_f64

pytestmark = pytest.mark.gpu


def layers(wl, dedup):
    w = [dev_bf16(synth.make_weight(wl, m)) for m in ("gate", "up", "down")]
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup)
    return moe.MoELayer(shape, *w, fuse_combine=True), moe.MoELayer(shape, *w)


@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("residual", [True, False])
@pytest.mark.parametrize("name", ["tiny", "ragged", "wide", "odd_h", "k_eq_e", "e256", "deep_k"])
def test_fused_combine_matches_oracle(name, residual, dedup):
    wl = SMALL[name]
    fused, plain = layers(wl, dedup)
    L, x = synth.make_logits(wl), synth.make_x(wl)
    res = synth.make_residual(wl) if residual else None
    args = (torch.from_numpy(L).cuda(), dev_bf16(x), None if res is None else dev_bf16(res))
    out_f = fused.forward(*args).clone()
    out_p = plain.forward(*args).clone()
    torch.cuda.synchronize()
    fused.check_device_errors()
    w = [synth.make_weight(wl, m) for m in ("gate", "up", "down")]
    ref = oracle.layer_forward(L, x, *w, wl.k, wl.W, residual=res, dedup=dedup)
    assert_close(host_f64(out_f), ref["out"], "fused combine")
    # the unfused layer rounds y to bf16 and sums in a fixed order; the two
    # agree to the same tolerance
    assert_close(host_f64(out_f), host_f64(out_p), "fused vs unfused")


def test_fused_combine_in_place_and_launch_count():
    wl = SMALL["ragged"]
    fused, _ = layers(wl, False)
    L, x, res = synth.make_logits(wl), synth.make_x(wl), synth.make_residual(wl)
    stream_buf = dev_bf16(res)
    fused.forward(torch.from_numpy(L).cuda(), dev_bf16(x), stream_buf, out=stream_buf)
    torch.cuda.synchronize()
    w = [synth.make_weight(wl, m) for m in ("gate", "up", "down")]
    ref = oracle.layer_forward(L, x, *w, wl.k, wl.W, residual=res)
    assert_close(host_f64(stream_buf), ref["out"], "in-place fused combine")
    assert fused.stage_names()[-1] == "down_combine"
    assert "combine" not in fused.stage_names() and "down" not in fused.stage_names()


def test_fused_combine_rejects_a_shared_expert():
    wl = SMALL["tiny"]
    w = [dev_bf16(synth.make_weight(wl, m)) for m in ("gate", "up", "down")]
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I)
    with pytest.raises(ValueError):
        moe.MoELayer(shape, *w, shared=tuple(w), fuse_combine=True)
