"""The packed weight layout (moe_pack_weights, MOE_WEIGHTS_PACKED): the packed
copies are exactly the blocks the header defines, and every GEMM path gives
the same bits on packed and row-major weights."""
import numpy as np
import pytest
import torch

from cases import SMALL
from combine_warp_top_gb300 import moe, synth
from gpu_util import dev_bf16, dev_i32, host_u16

pytestmark = pytest.mark.gpu


def packed_reference(w_gate, w_up, w_down, E, H, I):
    """The blocks of the header's definition, built with numpy: gate/up block
    (e, b, q) = rows 128b.. of w_gate then of w_up, columns 64q..; down block
    (e, b, q) = rows 256b.. of w_down, columns 64q..; zeros past the edges."""
    NBg, KBg = -(-I // 128), -(-H // 64)
    gu = np.zeros((E, NBg, KBg, 256, 64), np.uint16)
    g = np.zeros((E, NBg * 128, KBg * 64), np.uint16)
    u = np.zeros_like(g)
    g[:, :I, :H] = w_gate.reshape(E, I, H)
    u[:, :I, :H] = w_up.reshape(E, I, H)
    for b in range(NBg):
        for q in range(KBg):
            gu[:, b, q, :128] = g[:, 128 * b:128 * b + 128, 64 * q:64 * q + 64]
            gu[:, b, q, 128:] = u[:, 128 * b:128 * b + 128, 64 * q:64 * q + 64]
    NBd, KBd = -(-H // 256), -(-I // 64)
    dn = np.zeros((E, NBd, KBd, 256, 64), np.uint16)
    d = np.zeros((E, NBd * 256, KBd * 64), np.uint16)
    d[:, :H, :I] = w_down.reshape(E, H, I)
    for b in range(NBd):
        for q in range(KBd):
            dn[:, b, q] = d[:, 256 * b:256 * b + 256, 64 * q:64 * q + 64]
    return gu.reshape(-1), dn.reshape(-1)


@pytest.mark.parametrize("name", ["tiny", "ragged", "wide", "odd_h", "deep_k", "k32"])
def test_pack_matches_the_block_definition(name):
    wl = SMALL[name]
    wg, wu, wd = (synth.make_weight(wl, w) for w in ("gate", "up", "down"))
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I)
    gu, dn = moe.pack_weights(shape, dev_bf16(wg), dev_bf16(wu), dev_bf16(wd))
    torch.cuda.synchronize()
    ref_gu, ref_dn = packed_reference(wg, wu, wd, wl.E, wl.H, wl.I)
    assert gu.numel() * 2 == moe.moe_packed_gate_up_bytes(shape) == ref_gu.size * 2
    assert dn.numel() * 2 == moe.moe_packed_down_bytes(shape) == ref_dn.size * 2
    assert np.array_equal(host_u16(gu), ref_gu)
    assert np.array_equal(host_u16(dn), ref_dn)


def test_pack_one_output_only():
    wl = SMALL["ragged"]
    wg, wu, wd = (synth.make_weight(wl, w) for w in ("gate", "up", "down"))
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I)
    ref_gu, ref_dn = packed_reference(wg, wu, wd, wl.E, wl.H, wl.I)
    dn = torch.zeros(moe.moe_packed_down_bytes(shape) // 2, dtype=torch.bfloat16, device="cuda")
    moe.moe_pack_weights(None, None, dev_bf16(wd), shape, None, dn)
    gu = torch.zeros(moe.moe_packed_gate_up_bytes(shape) // 2, dtype=torch.bfloat16,
                     device="cuda")
    moe.moe_pack_weights(dev_bf16(wg), dev_bf16(wu), None, shape, gu, None)
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(dn), ref_dn)
    assert np.array_equal(host_u16(gu), ref_gu)


# the whole layer on both layouts: single-CTA (gathered plain rows), CTA pair
# (dispatched rows), dedup (gathered dedup rows), and the combine in the down
# epilogue; out, h and y must agree bit for bit (the fused combine's fp32
# atomics are compared within rounding instead)
@pytest.mark.parametrize("gemm", ["single", "pair"])
@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("name", ["ragged", "wide", "odd_h", "k12"])
def test_layer_bit_identical_on_packed_weights(name, dedup, gemm):
    wl = SMALL[name]
    wg, wu, wd = (dev_bf16(synth.make_weight(wl, w)) for w in ("gate", "up", "down"))
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup, gemm=gemm)
    placement = dev_i32(synth.permutation(0, 54, wl.E).astype(np.int32))
    L = torch.from_numpy(synth.make_logits(wl)).cuda()
    x = dev_bf16(synth.make_x(wl))
    res = dev_bf16(synth.make_residual(wl))
    outs = []
    for pack in (False, True):
        layer = moe.MoELayer(shape, wg, wu, wd, placement, pack=pack)
        assert layer.shape.weights == ("packed" if pack else "row_major")
        out = layer.forward(L, x, res).clone()
        torch.cuda.synchronize()
        layer.check_device_errors()
        outs.append((host_u16(out), host_u16(layer.h), host_u16(layer.y)))
    for a, b, what in zip(outs[0], outs[1], ("out", "h", "y")):
        assert np.array_equal(a, b), what


@pytest.mark.parametrize("name", ["ragged", "wide"])
def test_fused_combine_on_packed_weights(name):
    wl = SMALL[name]
    wg, wu, wd = (dev_bf16(synth.make_weight(wl, w)) for w in ("gate", "up", "down"))
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I)
    L = torch.from_numpy(synth.make_logits(wl)).cuda()
    x = dev_bf16(synth.make_x(wl))
    outs = []
    for pack in (False, True):
        layer = moe.MoELayer(shape, wg, wu, wd, fuse_combine=True, pack=pack)
        outs.append(layer.forward(L, x, None).float().clone())
        torch.cuda.synchronize()
        layer.check_device_errors()
    # fp32 atomics in tile-completion order: equal up to bf16 rounding steps
    diff = (outs[0] - outs[1]).abs().max().item()
    assert diff <= 2 ** -7 * outs[0].abs().max().item()
