"""Parity of the tcgen05 grouped SwiGLU FFN (moe_expert_ffn, through the C ABI)
against the float64 oracle: h and y over every row, on shapes that span
several 128x256 tiles, ragged expert segments and partial n/k blocks."""
import numpy as np
import pytest
import torch

import oracle
from cases import SMALL
from combine_warp_top_gb300 import moe, synth
from gpu_util import assert_close, dev_bf16, dev_i32, host_f64, host_u16

pytestmark = pytest.mark.gpu


def run_ffn(wl, dedup, ids=None, placement=None):
    if ids is None:
        ids, _ = oracle.route(synth.make_logits(wl), wl.k)
    pl = np.arange(wl.E) if placement is None else placement
    ref = oracle.dispatch_layout(ids, pl, wl.E, wl.W)
    x = synth.make_x(wl)
    wg, wu, wd = (synth.make_weight(wl, w) for w in ("gate", "up", "down"))
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup)
    lay = moe.Layout(shape)
    ws = moe.workspace(shape)
    moe.moe_dispatch_layout(dev_i32(ids), None if placement is None else dev_i32(placement),
                            shape, lay, ws)
    rows = shape.R_d_max if dedup else shape.R
    xd = torch.zeros(rows, wl.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch(dev_bf16(x), lay, shape, xd)
    h = torch.empty(shape.R, wl.I, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(shape.R, wl.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn(xd, lay, shape, dev_bf16(wg), dev_bf16(wu), dev_bf16(wd), None, h, y, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    xe_ref = oracle.dispatch(x, ref["row_token"])
    if dedup:
        # the materialised expansion is a bit-exact copy, and the expansion
        # done by the GEMM's gather warps (moe_expert_ffn) gives the same h
        xe = torch.empty(shape.R, wl.H, dtype=torch.bfloat16, device="cuda")
        moe.moe_expand(xd, lay, shape, xe)
        h2 = torch.empty_like(h)
        moe.moe_ffn_gate_up(xe, lay, shape, dev_bf16(wg), dev_bf16(wu), h2, ws)
        torch.cuda.synchronize()
        assert np.array_equal(host_u16(xe), xe_ref)
        assert torch.equal(h.view(torch.int16), h2.view(torch.int16))
    h_ref, y_ref = oracle.expert_ffn(xe_ref, ref["expert_offsets"], ref["expert_counts"], wg, wu, wd)
    return host_f64(h), host_f64(y), h_ref, y_ref


@pytest.mark.parametrize("name", list(SMALL))
def test_ffn_matches_oracle(name):
    h, y, h_ref, y_ref = run_ffn(SMALL[name], dedup=False)
    assert_close(h, h_ref, "h")
    assert_close(y, y_ref, "y")


@pytest.mark.parametrize("name", ["tiny", "wide", "odd_h"])
def test_ffn_after_dedup_expansion(name):
    h, y, h_ref, y_ref = run_ffn(SMALL[name], dedup=True)
    assert_close(h, h_ref, "h")
    assert_close(y, y_ref, "y")


def test_ffn_per_expert_segments():
    """Each expert segment individually (catches rows attributed to the wrong
    expert, which a global norm could hide)."""
    wl = SMALL["ragged"]
    ids, _ = oracle.route(synth.make_logits(wl), wl.k)
    ref = oracle.dispatch_layout(ids, np.arange(wl.E), wl.E, wl.W)
    h, y, h_ref, y_ref = run_ffn(wl, dedup=False, ids=ids)
    for e in range(wl.E):
        a, n = ref["expert_offsets"][e], ref["expert_counts"][e]
        if n:
            assert_close(y[a:a + n], y_ref[a:a + n], f"y of expert {e}")


def test_ffn_skewed_and_tiny_segments():
    """One expert takes nearly every token (many m-blocks), others 0, 1 or 3 rows."""
    wl = synth.Workload("skew", 700, 256, 8, 2, 256, 2)
    ids = np.zeros((wl.N, 2), np.int32)
    ids[:, 0] = 3
    ids[:, 1] = 6
    ids[0, 1], ids[1, 1], ids[2, 1], ids[3, 1] = 1, 2, 2, 2
    ids[4, 1] = 0
    h, y, h_ref, y_ref = run_ffn(wl, dedup=False, ids=ids)
    assert_close(h, h_ref, "h")
    assert_close(y, y_ref, "y")


def test_ffn_permuted_placement():
    wl = synth.Workload("perm", 400, 256, 16, 4, 256, 4)
    ids, _ = oracle.route(synth.make_logits(wl), wl.k)
    placement = synth.permutation(0, 52, wl.E).astype(np.int32)
    h, y, h_ref, y_ref = run_ffn(wl, dedup=False, ids=ids, placement=placement)
    assert_close(y, y_ref, "y")


@pytest.mark.parametrize("name", ["tiny", "ragged", "wide", "odd_h", "deep_k", "e256"])
def test_gathered_rows_equal_dispatched_rows(name):
    """The gate/up GEMM fed by gather4 straight from x through row_token gives
    bit for bit the h of the GEMM fed by the dispatched rows."""
    wl = SMALL[name]
    ids, _ = oracle.route(synth.make_logits(wl), wl.k)
    x = dev_bf16(synth.make_x(wl))
    wg, wu = dev_bf16(synth.make_weight(wl, "gate")), dev_bf16(synth.make_weight(wl, "up"))
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I)
    lay = moe.Layout(shape)
    ws = moe.workspace(shape)
    moe.moe_dispatch_layout(dev_i32(ids), None, shape, lay, ws)
    xd = torch.empty(shape.R, wl.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch(x, lay, shape, xd)
    h1 = torch.empty(shape.R, wl.I, dtype=torch.bfloat16, device="cuda")
    h2 = torch.empty_like(h1)
    moe.moe_ffn_gate_up(xd, lay, shape, wg, wu, h1, ws)
    moe.moe_ffn_gate_up_gather(x, lay["row_token"], lay, shape, wg, wu, h2, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))
