"""The expert FFN with h kept on chip (moe_ffn_fused, gemm "fused"): the layer
against the oracle's forward pass, and y bit for bit against the two-kernel
path (same h rounding, same fp32 accumulation orders), on every small shape
with H <= 256 and on ragged I >= 1024 (the wide, 128-column-chunk form),
plain and dedup, row-major and packed weights; a shape with
several tiles per CTA and many chunks of I checked on every (expert, 128-row
tile) and on every segment's last row; the direct call on materialised rows
and through an index; the microbatch pipeline."""
import numpy as np
import pytest
import torch

import oracle
from cases import SMALL
from combine_warp_top_gb300 import moe, synth
from gpu_util import assert_close, dev_bf16, dev_i32, host_f64, host_u16

pytestmark = pytest.mark.gpu

FUSABLE = [n for n, wl in SMALL.items() if wl.H <= 256]


def run_layer(wl, w, gemm, dedup, pack, placement=None, residual=True, seed=0):
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup, gemm=gemm)
    layer = moe.MoELayer(shape, *w, placement, pack=pack)
    L = torch.from_numpy(synth.make_logits(wl, seed=seed)).cuda()
    x = dev_bf16(synth.make_x(wl, seed=seed))
    res = dev_bf16(synth.make_residual(wl, seed=seed)) if residual else None
    out = layer.forward(L, x, res).clone()
    torch.cuda.synchronize()
    layer.check_device_errors()
    return layer, out


@pytest.mark.parametrize("pack", [False, True])
@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("name", FUSABLE)
def test_fused_layer_against_oracle_and_two_kernels(name, dedup, pack):
    wl = SMALL[name]
    wh = [synth.make_weight(wl, m) for m in ("gate", "up", "down")]
    w = [dev_bf16(a) for a in wh]
    placement = synth.permutation(3, 55, wl.E).astype(np.int32) if wl.E > 1 else None
    pl = None if placement is None else dev_i32(placement)
    fused, out = run_layer(wl, w, "fused", dedup, pack, pl)
    assert fused.fused_ffn and "ffn" in fused.stage_names()
    assert fused.kernel_launches_per_step() == moe.MoELayer(
        moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup, gemm="single"), *w, pl,
        pack=False).kernel_launches_per_step() - 1
    # the automatic choice (the fused kernel or the two GEMMs, by the shape):
    # the same bits either way
    auto, out_a = run_layer(wl, w, "auto", dedup, pack, pl)
    assert auto.fused_ffn == moe.moe_layer_fuses_ffn(
        moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup))
    assert torch.equal(out.view(torch.int16), out_a.view(torch.int16))
    ref = oracle.layer_forward(synth.make_logits(wl), synth.make_x(wl), *wh, wl.k, wl.W,
                               placement=placement, residual=synth.make_residual(wl), dedup=dedup)
    assert np.array_equal(fused.topk_ids.view(wl.N, wl.k).cpu().numpy(), ref["topk_ids"])
    assert_close(host_f64(out), ref["out"], f"{name} fused out")
    single, out_s = run_layer(wl, w, "single", dedup, pack, pl)
    R = wl.N * wl.k
    assert np.array_equal(host_u16(fused.y[:R]), host_u16(single.y[:R])), "y"
    assert torch.equal(out.view(torch.int16), out_s.view(torch.int16))


# I >= 1024 runs the wide form (128-column chunks of I): ragged I with an odd
# number of 64-column down k-blocks (1032: the last chunk has one), a partial
# last chunk (1096), H = 256 (three ring stages) and a small H
WIDE = [synth.Workload("wide_i1032", 300, 200, 8, 2, 1032, 4),
        synth.Workload("wide_i1096", 257, 256, 6, 3, 1096, 3),
        synth.Workload("wide_i1408_h64", 500, 64, 16, 4, 1408, 4)]


@pytest.mark.parametrize("pack", [False, True])
@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("wl", WIDE, ids=lambda w: w.name)
def test_fused_wide_form_against_oracle_and_two_kernels(wl, dedup, pack):
    wh = [synth.make_weight(wl, m) for m in ("gate", "up", "down")]
    w = [dev_bf16(a) for a in wh]
    fused, out = run_layer(wl, w, "fused", dedup, pack)
    ref = oracle.layer_forward(synth.make_logits(wl), synth.make_x(wl), *wh, wl.k, wl.W,
                               residual=synth.make_residual(wl), dedup=dedup)
    assert_close(host_f64(out), ref["out"], f"{wl.name} fused out")
    single, out_s = run_layer(wl, w, "single", dedup, pack)
    R = wl.N * wl.k
    assert np.array_equal(host_u16(fused.y[:R]), host_u16(single.y[:R])), "y"
    assert torch.equal(out.view(torch.int16), out_s.view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "odd_h", "k32"])
def test_fused_moe_delta_alone(name):
    wl = SMALL[name]
    wh = [synth.make_weight(wl, m) for m in ("gate", "up", "down")]
    _, out = run_layer(wl, [dev_bf16(a) for a in wh], "fused", False, True, residual=False)
    ref = oracle.layer_forward(synth.make_logits(wl), synth.make_x(wl), *wh, wl.k, wl.W)
    assert_close(host_f64(out), ref["out"], f"{name} fused delta")


# 16384 tokens, top-4 of 16 experts: 512 tiles of 128 rows over at most one CTA
# per SM (several tiles per CTA), 22 chunks of I = 1408 (the correlated
# workloads' width), H = 256 (the largest the fused kernel takes: 3 ring stages)
MANY = synth.Workload("fused_many", 16384, 256, 16, 4, 1408, 4)


@pytest.mark.parametrize("H", [256, 64])
def test_fused_many_tiles_every_tile_checked(H):
    wl = synth.Workload(MANY.name, MANY.N, H, MANY.E, MANY.k, MANY.I, MANY.W)
    w = [synth.make_weight_device(wl, m) for m in ("gate", "up", "down")]
    fused, out = run_layer(wl, w, "fused", False, True)
    single, out_s = run_layer(wl, w, "single", False, True)
    R = wl.N * wl.k
    assert torch.equal(fused.y[:R].view(torch.int16), single.y[:R].view(torch.int16))
    assert torch.equal(out.view(torch.int16), out_s.view(torch.int16))
    # oracle: one row in every (expert, 128-row tile) and every segment's last row
    L, x, res = synth.make_logits(wl), synth.make_x(wl), synth.make_residual(wl)
    ids, tw = oracle.route(L, wl.k)
    lay = oracle.dispatch_layout(ids, np.arange(wl.E), wl.E, wl.W)
    off, cnt = lay["expert_offsets"], lay["expert_counts"]
    rows = []
    for e in range(wl.E):
        for r0 in range(0, int(cnt[e]), 128):
            rows.append(int(off[e]) + r0 + (r0 // 128 * 37) % min(128, int(cnt[e]) - r0))
        if cnt[e]:
            rows.append(int(off[e]) + int(cnt[e]) - 1)
    toks = np.unique(lay["row_token"][np.array(rows)]).astype(np.int64)

    def weights_of(e):
        return tuple(synth.make_weight(wl, m, experts=[e])[0] for m in ("gate", "up", "down"))

    want, y_want = oracle.token_outputs(x[toks], ids[toks], tw[toks], weights_of, res[toks])
    assert_close(host_f64(out[torch.from_numpy(toks).cuda()]), want, "out")
    pr = lay["pair_row"][toks].reshape(-1).astype(np.int64)
    assert_close(host_f64(fused.y[torch.from_numpy(pr).cuda()]), y_want.reshape(-1, H), "y rows")


def test_fused_call_on_materialised_and_indexed_rows():
    """moe_ffn_fused on the dispatched rows (row_index NULL) and on x through
    row_token give the same y bits as moe_ffn_gate_up + moe_ffn_down."""
    wl = SMALL["ragged"]
    w = [dev_bf16(synth.make_weight(wl, m)) for m in ("gate", "up", "down")]
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I)
    R = shape.R
    lay, ws = moe.Layout(shape), moe.workspace(shape)
    ids = torch.empty(R, dtype=torch.int32, device="cuda")
    tw = torch.empty(R, dtype=torch.float32, device="cuda")
    x = dev_bf16(synth.make_x(wl))
    moe.moe_route(torch.from_numpy(synth.make_logits(wl)).cuda(), shape, ids, tw)
    moe.moe_dispatch_layout(ids, None, shape, lay, ws)
    xd = torch.empty(R, wl.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch(x, lay, shape, xd)
    h = torch.empty(R, wl.I, dtype=torch.bfloat16, device="cuda")
    y_ref = torch.empty(R, wl.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_ffn_gate_up(xd, lay, shape, w[0], w[1], h, ws)
    moe.moe_ffn_down(h, lay, shape, w[2], y_ref, ws)
    y1 = torch.full((R, wl.H), 7.0, dtype=torch.bfloat16, device="cuda")
    y2 = torch.full((R, wl.H), 7.0, dtype=torch.bfloat16, device="cuda")
    moe.moe_ffn_fused(xd, None, lay, shape, *w, y1, ws)
    moe.moe_ffn_fused(x, lay["row_token"], lay, shape, *w, y2, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    assert torch.equal(y1.view(torch.int16), y_ref.view(torch.int16))
    assert torch.equal(y2.view(torch.int16), y_ref.view(torch.int16))
    # moe_expert_ffn with gemm "fused" is the same call; h is not needed
    fshape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, gemm="fused")
    y3 = torch.zeros(R, wl.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn(xd, lay, fshape, *w, None, h, y3, ws)
    torch.cuda.synchronize()
    assert torch.equal(y3.view(torch.int16), y_ref.view(torch.int16))
    # a shape wider than the TMEM tile is refused before any launch
    wide = moe.Shape(wl.N, 264, wl.E, wl.k, wl.W, wl.I)
    with pytest.raises(moe.MoeError, match="UNSUPPORTED"):
        moe.moe_ffn_fused(torch.empty(R, 264, dtype=torch.bfloat16, device="cuda"), None,
                          moe.Layout(wide), wide, *(torch.empty(wl.E * 264 * wl.I,
                                                                dtype=torch.bfloat16,
                                                                device="cuda")
                                                    for _ in range(3)),
                          torch.empty(R, 264, dtype=torch.bfloat16, device="cuda"),
                          moe.workspace(wide))


@pytest.mark.parametrize("dedup", [False, True])
def test_fused_pipeline_is_bit_identical(dedup):
    wl = SMALL["ragged"]
    wh = [synth.make_weight(wl, m) for m in ("gate", "up", "down")]
    w = tuple(dev_bf16(a) for a in wh)
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup, gemm="fused")
    layer = moe.MoELayer(shape, *w)
    pipe = moe.MicrobatchPipeline(shape, *w, microbatch=77)
    Lh, xh, rh = synth.make_logits(wl), synth.make_x(wl), synth.make_residual(wl)
    L = torch.from_numpy(Lh).cuda()
    x, res = dev_bf16(xh), dev_bf16(rh)
    want = layer.forward(L, x, res).clone()
    got = pipe.forward(L, x, res)
    torch.cuda.synchronize()
    pipe.check_device_errors()
    ref = oracle.layer_forward(Lh, xh, *wh, wl.k, wl.W, residual=rh, dedup=dedup)
    assert_close(host_f64(got), ref["out"], "fused pipeline out")
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
