"""Bounds checks of the CUDA path by guard bands.

Every buffer handed to the C ABI is a view into a larger device allocation
whose bytes before and after the view (the guards) hold a fill pattern.  After
a run the tests check that

* every guard still holds the pattern (no write before or after any buffer),
* every input (logits, x, weights, residual, placement) is unchanged, bit for
  bit, guards included,
* rows a call must leave alone are untouched: the dedup rows past R_d of xd
  and of the partial buffer, the dedup_row_token entries past R_d, and the
  whole xd buffer when the layer gathers its plain rows inside the gate/up GEMM,
* and the outputs match the oracle (so that the run did its work).

The shapes are the ragged and edge shapes of the other parity tests (segments
that end inside a tile, widths below one TMA box, one token, one expert, the
largest k), each with and without dedup, on both GEMM kernels.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from cases import SMALL
from combine_warp_top_gb300 import moe, synth
from gpu_util import assert_close, host_f64

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes of guard on each side (keeps every view 256-byte aligned)
FILL = 0xA5           # guard byte: bf16 0xA5A5 = -2.9e-16, int32 0xA5A5A5A5 < 0

EDGE = [
    synth.Workload("one_token", 1, 256, 8, 2, 128, 2),
    synth.Workload("one_expert", 300, 128, 1, 1, 128, 1),
    synth.Workload("narrow8", 130, 8, 4, 2, 8, 4),
    synth.Workload("wide_i_small_h", 300, 64, 4, 2, 1000, 2),
]
SHAPES = [SMALL[n] for n in ("ragged", "odd_h", "k12", "k32", "e256")] + EDGE


class Guarded:
    """A view of `n` elements of `dtype` with GUARD bytes of FILL on each side."""

    def __init__(self, n, dtype, data=None, zero=False):
        self.esize = torch.empty(0, dtype=dtype).element_size()
        self.n = max(int(n), 1)
        self.raw = torch.full((2 * GUARD + self.n * self.esize,), FILL, dtype=torch.uint8,
                              device="cuda")
        self.view = self.raw[GUARD:GUARD + self.n * self.esize].view(dtype)
        if zero:
            self.view.zero_()
        if data is not None:
            self.view[:data.numel()].copy_(data.reshape(-1))
        self.before = None

    def snapshot(self):
        self.before = self.raw.clone()

    def guards_intact(self):
        lo = self.raw[:GUARD]
        hi = self.raw[GUARD + self.n * self.esize:]
        return bool((lo == FILL).all()) and bool((hi == FILL).all())

    def unchanged(self):
        return bool(torch.equal(self.raw, self.before))

    def untouched(self, first, last):
        """Elements [first, last) of the view still hold the fill pattern."""
        if last <= first:
            return True
        b = self.raw[GUARD + first * self.esize:GUARD + last * self.esize]
        return bool((b == FILL).all())


class GuardedLayout:
    """A moe_layout whose arrays are guarded views (duck-types moe.Layout)."""

    def __init__(self, shape):
        self.shape = shape
        N, E, k, W = shape.N, shape.E, shape.k, shape.W
        sizes = dict(expert_counts=E, expert_offsets=E + 1, rank_offsets=W + 1,
                     row_token=N * k, pair_row=N * k)
        if shape.dedup:
            sizes.update(dedup_counts=W, dedup_offsets=W + 1, dedup_row_token=N * min(k, W),
                         pair_dedup_row=N * k, expand_src=N * k, n_dedup_rows=1)
        self.g = {n: Guarded(s, torch.int32) for n, s in sizes.items()}
        self.tensors = {n: g.view for n, g in self.g.items()}
        self.c = moe.MoeLayout(*[ctypes.c_void_p(self.tensors[n].data_ptr())
                                 if n in self.tensors else None for n in moe.LAYOUT_FIELDS])

    def __getitem__(self, name):
        return self.tensors[name]


def bf16_of(a_u16):
    return torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).view(torch.bfloat16)


def inputs(wl, shape):
    """Guarded device inputs and their host copies."""
    Lh, xh, rh = synth.make_logits(wl), synth.make_x(wl), synth.make_residual(wl)
    wh = [synth.make_weight(wl, m) for m in ("gate", "up", "down")]
    d = dict(
        logits=Guarded(wl.N * wl.E, torch.float32, torch.from_numpy(Lh)),
        x=Guarded(wl.N * wl.H, torch.bfloat16, bf16_of(xh)),
        residual=Guarded(wl.N * wl.H, torch.bfloat16, bf16_of(rh)),
        w_gate=Guarded(wh[0].size, torch.bfloat16, bf16_of(wh[0])),
        w_up=Guarded(wh[1].size, torch.bfloat16, bf16_of(wh[1])),
        w_down=Guarded(wh[2].size, torch.bfloat16, bf16_of(wh[2])),
    )
    for g in d.values():
        g.snapshot()
    return d, (Lh, xh, rh, wh)


def outputs(shape):
    s = shape
    return dict(
        topk_ids=Guarded(s.R, torch.int32),
        topk_w=Guarded(s.R, torch.float32),
        xd=Guarded((s.R_d_max if s.dedup else s.R) * s.H, torch.bfloat16),
        xe=Guarded(s.R * s.H, torch.bfloat16),
        h=Guarded(s.R * s.I, torch.bfloat16),
        y=Guarded(s.R * s.H, torch.bfloat16),
        partial=Guarded(s.R_d_max * s.H, torch.bfloat16),
        out=Guarded(s.N * s.H, torch.bfloat16),
        acc=Guarded(s.N * s.H, torch.float32),
        ws=Guarded(moe.moe_workspace_bytes(s), torch.uint8, zero=True),
    )


def check_guards(named):
    bad = [n for n, g in named.items() if not g.guards_intact()]
    assert not bad, f"guard bands overwritten: {bad}"


def check_common(shape, ins, outs, lay, wl):
    check_guards(ins)
    check_guards(outs)
    check_guards(lay.g)
    changed = [n for n, g in ins.items() if not g.unchanged()]
    assert not changed, f"inputs modified: {changed}"
    ids = outs["topk_ids"].view.cpu().numpy()
    assert ids.min() >= 0 and ids.max() < wl.E
    if shape.dedup:
        Rd = int(lay["n_dedup_rows"][0].item())
        assert shape.N <= Rd <= shape.R_d_max
        assert lay.g["dedup_row_token"].untouched(Rd, shape.R_d_max)
        assert outs["xd"].untouched(Rd * shape.H, shape.R_d_max * shape.H)
        return Rd
    return None


def as_bf16(g, rows, cols):
    return g.view[:rows * cols].view(rows, cols)


@pytest.mark.parametrize("gemm", ["auto", "single", "pair"])
@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("wl", SHAPES, ids=lambda w: w.name)
def test_layer_forward_stays_in_bounds(wl, dedup, gemm):
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup, gemm=gemm)
    ins, (Lh, xh, rh, wh) = inputs(wl, shape)
    # the dedup runs place the experts by a seeded permutation, the plain ones
    # contiguously (placement = NULL)
    placement = np.random.default_rng(wl.E).permutation(wl.E).astype(np.int32) if dedup else None
    if placement is not None:
        ins["placement"] = Guarded(wl.E, torch.int32, torch.from_numpy(placement))
        ins["placement"].snapshot()
    outs = outputs(shape)
    lay = GuardedLayout(shape)
    moe.moe_layer_forward(ins["logits"].view, ins["x"].view,
                          None if placement is None else ins["placement"].view, ins["w_gate"].view,
                          ins["w_up"].view, ins["w_down"].view, ins["residual"].view, shape,
                          outs["topk_ids"].view, outs["topk_w"].view, lay, outs["xd"].view,
                          None, outs["h"].view, outs["y"].view, None, outs["out"].view,
                          outs["ws"].view)
    torch.cuda.synchronize()
    assert moe.moe_get_error(outs["ws"].view) == 0
    check_common(shape, ins, outs, lay, wl)
    if moe.moe_layer_skips_dispatch(shape):
        # the plain rows were gathered inside the GEMM: xd is never written
        assert outs["xd"].untouched(0, shape.R * shape.H)
    if moe.moe_layer_fuses_ffn(shape):
        # the fused expert FFN (the default for small H) keeps h on chip
        assert outs["h"].untouched(0, outs["h"].n)
    for n in ("xe", "partial", "acc"):
        assert outs[n].untouched(0, outs[n].n), n
    ref = oracle.layer_forward(Lh, xh, *wh, wl.k, wl.W, placement=placement, residual=rh,
                               dedup=dedup)
    assert_close(host_f64(as_bf16(outs["out"], wl.N, wl.H)), ref["out"], "out")


@pytest.mark.parametrize("wl", SHAPES, ids=lambda w: w.name)
def test_materialised_dedup_stages_stay_in_bounds(wl):
    """The dedup layer as separate calls with every intermediate written: the
    expansion into xe, the gate/up GEMM on xe, and the two-level combine
    through the partial buffer."""
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=True)
    ins, (Lh, xh, rh, wh) = inputs(wl, shape)
    outs = outputs(shape)
    lay = GuardedLayout(shape)
    ws = outs["ws"].view
    moe.moe_route(ins["logits"].view, shape, outs["topk_ids"].view, outs["topk_w"].view)
    moe.moe_dispatch_layout(outs["topk_ids"].view, None, shape, lay, ws)
    moe.moe_dispatch(ins["x"].view, lay, shape, outs["xd"].view)
    moe.moe_expand(outs["xd"].view, lay, shape, outs["xe"].view)
    moe.moe_ffn_gate_up(outs["xe"].view, lay, shape, ins["w_gate"].view, ins["w_up"].view,
                        outs["h"].view, ws)
    moe.moe_ffn_down(outs["h"].view, lay, shape, ins["w_down"].view, outs["y"].view, ws)
    moe.moe_combine(outs["y"].view, outs["topk_w"].view, lay, shape, outs["partial"].view,
                    ins["residual"].view, outs["out"].view)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    Rd = check_common(shape, ins, outs, lay, wl)
    assert outs["partial"].untouched(Rd * shape.H, shape.R_d_max * shape.H)
    ref = oracle.layer_forward(Lh, xh, *wh, wl.k, wl.W, residual=rh, dedup=True)
    assert_close(host_f64(as_bf16(outs["out"], wl.N, wl.H)), ref["out"], "out")
    assert_close(host_f64(as_bf16(outs["partial"], Rd, wl.H)), ref["partial"], "partial")


@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("wl", SHAPES, ids=lambda w: w.name)
def test_fused_combine_stays_in_bounds(wl, dedup):
    """The down GEMM with the combine in its epilogue: the fp32 accumulator is
    written only inside its [N, H] view, y is never written."""
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup)
    ins, (Lh, xh, rh, wh) = inputs(wl, shape)
    outs = outputs(shape)
    lay = GuardedLayout(shape)
    ws = outs["ws"].view
    moe.moe_route(ins["logits"].view, shape, outs["topk_ids"].view, outs["topk_w"].view)
    moe.moe_dispatch_layout(outs["topk_ids"].view, None, shape, lay, ws)
    moe.moe_dispatch(ins["x"].view, lay, shape, outs["xd"].view)
    if dedup:
        moe.moe_ffn_gate_up_gather(outs["xd"].view, lay["expand_src"], lay, shape,
                                   ins["w_gate"].view, ins["w_up"].view, outs["h"].view, ws)
    else:
        moe.moe_ffn_gate_up(outs["xd"].view, lay, shape, ins["w_gate"].view, ins["w_up"].view,
                            outs["h"].view, ws)
    moe.moe_ffn_down_combine(outs["h"].view, outs["topk_w"].view, lay, shape,
                             ins["w_down"].view, ins["residual"].view, outs["acc"].view,
                             outs["out"].view, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    check_common(shape, ins, outs, lay, wl)
    assert outs["y"].untouched(0, outs["y"].n)
    ref = oracle.layer_forward(Lh, xh, *wh, wl.k, wl.W, residual=rh, dedup=dedup)
    assert_close(host_f64(as_bf16(outs["out"], wl.N, wl.H)), ref["out"], "out")
