"""The CTA-pair (tcgen05 cta_group::2, 256-row tiles) grouped GEMMs, chosen
through the shape's gemm field, against the oracle and bit for bit against the
single-CTA kernels (same K order of accumulation)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from cases import SMALL
from combine_warp_top_gb300 import moe, synth
from gpu_util import assert_close, dev_bf16, dev_i32, host_f64

pytestmark = pytest.mark.gpu


def ffn_outputs(wl, pair, ids=None):
    if ids is None:
        ids, _ = oracle.route(synth.make_logits(wl), wl.k)
    x = synth.make_x(wl)
    w = [synth.make_weight(wl, m) for m in ("gate", "up", "down")]
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, gemm="pair" if pair else "single")
    lay = moe.Layout(shape)
    ws = moe.workspace(shape)
    moe.moe_dispatch_layout(dev_i32(ids), None, shape, lay, ws)
    xd = torch.empty(shape.R, wl.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch(dev_bf16(x), lay, shape, xd)
    h = torch.empty(shape.R, wl.I, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(shape.R, wl.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn(xd, lay, shape, *[dev_bf16(a) for a in w], None, h, y, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    ref = oracle.dispatch_layout(ids, np.arange(wl.E), wl.E, wl.W)
    return h, y, ids, ref, x, w


@pytest.mark.parametrize("name", ["tiny", "ragged", "wide", "odd_h", "deep_k", "e256", "k_eq_e"])
def test_pair_kernel_matches_oracle_and_single_cta(name):
    wl = SMALL[name]
    h2, y2, ids, ref, x, w = ffn_outputs(wl, True)
    h_ref, y_ref = oracle.expert_ffn(oracle.dispatch(x, ref["row_token"]), ref["expert_offsets"],
                                     ref["expert_counts"], *w)
    assert_close(host_f64(h2), h_ref, "h")
    assert_close(host_f64(y2), y_ref, "y")
    h1, y1, *_ = ffn_outputs(wl, False, ids=ids)
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_pair_kernel_skewed_segments():
    """One expert with many 256-row tiles, others with 0, 1, 3 rows or a few
    hundred (ragged halves of a pair tile on either CTA)."""
    wl = synth.Workload("skew", 1500, 256, 8, 2, 384, 2)
    ids = np.zeros((wl.N, 2), np.int32)
    ids[:, 0] = 3
    ids[:, 1] = 6
    ids[:130, 1] = 5          # 130 rows: the peer CTA's half of the tile is ragged
    ids[130:400, 1] = 1       # 270 rows: two tiles, the second mostly empty
    ids[400, 1], ids[401:404, 1] = 0, 2
    h2, y2, ids, ref, x, w = ffn_outputs(wl, True, ids=ids)
    h1, y1, *_ = ffn_outputs(wl, False, ids=ids)
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    h_ref, y_ref = oracle.expert_ffn(oracle.dispatch(x, ref["row_token"]), ref["expert_offsets"],
                                     ref["expert_counts"], *w)
    assert_close(host_f64(y2), y_ref, "y")


@pytest.mark.parametrize("dedup", [False, True])
def test_pair_layer_with_shared_expert(dedup):
    wl = SMALL["wide"]
    w = [synth.make_weight(wl, m) for m in ("gate", "up", "down")]
    one = synth.Workload("s", wl.N, wl.H, 1, 1, 256, 1)
    sh = tuple(synth.make_weight(one, m, seed=3)[0] for m in ("gate", "up", "down"))
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup, gemm="pair")
    layer = moe.MoELayer(shape, *[dev_bf16(a) for a in w], shared=tuple(dev_bf16(a) for a in sh))
    L, x, res = synth.make_logits(wl), synth.make_x(wl), synth.make_residual(wl)
    out = layer.forward(torch.from_numpy(L).cuda(), dev_bf16(x), dev_bf16(res))
    torch.cuda.synchronize()
    layer.check_device_errors()
    ref = oracle.layer_forward(L, x, *w, wl.k, wl.W, residual=res, dedup=dedup, shared=sh)
    assert_close(host_f64(out), ref["out"], "out")


@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("name", ["tiny", "ragged", "wide", "odd_h", "deep_k", "e256"])
def test_gathered_rows_equal_dispatched_rows(name, dedup):
    """Both kernels fed by their gather warps (rows of x through row_token, or
    of the dedup rows through expand_src) give bit for bit the h of the same
    kernel fed by materialised rows: the gather changes only how A reaches
    shared memory."""
    wl = SMALL[name]
    ids, _ = oracle.route(synth.make_logits(wl), wl.k)
    x = dev_bf16(synth.make_x(wl))
    wg, wu = dev_bf16(synth.make_weight(wl, "gate")), dev_bf16(synth.make_weight(wl, "up"))
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup)
    lay = moe.Layout(shape)
    ws = moe.workspace(shape)
    moe.moe_dispatch_layout(dev_i32(ids), None, shape, lay, ws)
    xd = torch.empty(shape.R_d_max if dedup else shape.R, wl.H, dtype=torch.bfloat16,
                     device="cuda")
    moe.moe_dispatch(x, lay, shape, xd)
    if dedup:
        rows = torch.empty(shape.R, wl.H, dtype=torch.bfloat16, device="cuda")
        moe.moe_expand(xd, lay, shape, rows)
        src, index = xd, lay["expand_src"]
    else:
        rows, src, index = xd, x, lay["row_token"]
    outs = {}
    for pair in ("single", "pair"):
        s = dataclasses.replace(shape, gemm=pair)
        h_rows = torch.empty(shape.R, wl.I, dtype=torch.bfloat16, device="cuda")
        h_gather = torch.empty_like(h_rows)
        moe.moe_ffn_gate_up(rows, lay, s, wg, wu, h_rows, ws)
        moe.moe_ffn_gate_up_gather(src, index, lay, s, wg, wu, h_gather, ws)
        torch.cuda.synchronize()
        assert moe.moe_get_error(ws) == 0
        assert torch.equal(h_rows.view(torch.int16), h_gather.view(torch.int16)), pair
        outs[pair] = h_gather
    assert torch.equal(outs["single"].view(torch.int16), outs["pair"].view(torch.int16))
