"""Host logic of the layer wrapper, without a GPU: which stages MoELayer runs
for a shape (and so which stages the bench times and the launch count it
claims) follows the library's own choices -- moe_layer_skips_dispatch and
moe_layer_fuses_ffn, both functions of the shape alone.  The layers here are
built on CPU tensors with pack=False, so nothing is launched."""
import pytest
import torch

from combine_warp_top_gb300 import moe


def layer(shape, fuse_combine=False, shared=None):
    E, H, I = shape.E, shape.H, shape.I
    bf = dict(dtype=torch.bfloat16, device="cpu")
    w = (torch.zeros(E, I, H, **bf), torch.zeros(E, I, H, **bf), torch.zeros(E, H, I, **bf))
    return moe.MoELayer(shape, *w, device="cpu", pack=False, fuse_combine=fuse_combine,
                        shared=shared)


@pytest.mark.parametrize("shape,stages", [
    # small H: the expert FFN is the one fused kernel, plain rows gathered from x
    (moe.Shape(64, 128, 8, 2, 2, 256), ["route", "layout", "ffn", "combine"]),
    # dedup: the dedup rows are dispatched first, then expanded by the fused kernel
    (moe.Shape(64, 128, 8, 2, 2, 256, dedup=True),
     ["route", "layout", "dispatch", "ffn", "combine"]),
    # H > 256, few rows per expert: single-CTA GEMMs, dispatch fused into gate/up
    (moe.Shape(4096, 7168, 256, 8, 8, 2048), ["route", "layout", "gate_up", "down", "combine"]),
    # H <= 256 without dedup: fused by default; with dedup only up to H = 128
    (moe.Shape(4096, 256, 8, 2, 4, 384), ["route", "layout", "ffn", "combine"]),
    # few rows (N*k < 4096) and I > 256: the two GEMMs
    (moe.Shape(300, 256, 8, 2, 4, 384), ["route", "layout", "gate_up", "down", "combine"]),
    (moe.Shape(300, 256, 8, 2, 4, 384, dedup=True),
     ["route", "layout", "dispatch", "gate_up", "down", "combine"]),
    # many rows per expert: the CTA-pair GEMMs, which have no gather mode
    (moe.Shape(8192, 4096, 8, 2, 8, 14336),
     ["route", "layout", "dispatch", "gate_up", "down", "combine"]),
    # the two GEMMs named explicitly at H = 128
    (moe.Shape(64, 128, 8, 2, 2, 256, gemm="single"),
     ["route", "layout", "gate_up", "down", "combine"]),
    # the fused kernel named explicitly on a dedup layer at H = 256
    (moe.Shape(300, 256, 8, 2, 4, 384, dedup=True, gemm="fused"),
     ["route", "layout", "dispatch", "ffn", "combine"]),
])
def test_stages_follow_the_library(shape, stages):
    lay = layer(shape)
    assert lay.stage_names() == stages
    assert lay.fused_ffn == ("ffn" in stages) == moe.moe_layer_fuses_ffn(shape)
    assert lay.fused_dispatch == ("dispatch" not in stages) == moe.moe_layer_skips_dispatch(shape)


def test_launch_counts():
    """route 1 + layout (1 for one block of 256 tokens, else 2, or 3 with a
    separate scan) + dispatch (unless gathered) + FFN (1 fused, 2 as two
    GEMMs) + combine 1."""
    fused = layer(moe.Shape(64, 128, 8, 2, 2, 256))
    two = layer(moe.Shape(64, 128, 8, 2, 2, 256, gemm="single"))
    assert fused.kernel_launches_per_step() == 1 + 1 + 0 + 1 + 1
    assert two.kernel_launches_per_step() == 1 + 1 + 0 + 2 + 1
    dedup = layer(moe.Shape(257, 128, 8, 2, 2, 256, dedup=True))  # two layout blocks
    assert dedup.kernel_launches_per_step() == 1 + 2 + 1 + 1 + 1
    big = layer(moe.Shape(70000, 128, 64, 6, 32, 256))  # count tables over 64 KB: a scan launch
    assert moe.layout_launches(big.shape) == 3
    assert big.kernel_launches_per_step() == 1 + 3 + 0 + 1 + 1


def test_fused_combine_keeps_the_two_gemms():
    """The combine in the down GEMM's epilogue needs a down GEMM: with it the
    layer runs gate/up + down_combine even where it would fuse the FFN, and a
    shape that names the fused kernel is refused."""
    lay = layer(moe.Shape(64, 128, 8, 2, 2, 256), fuse_combine=True)
    assert not lay.fused_ffn
    assert lay.stage_names() == ["route", "layout", "gate_up", "down_combine"]
    with pytest.raises(ValueError):
        layer(moe.Shape(64, 128, 8, 2, 2, 256, gemm="fused"), fuse_combine=True)


def test_shared_expert_stage():
    bf = dict(dtype=torch.bfloat16, device="cpu")
    sh = (torch.zeros(64, 128, **bf), torch.zeros(64, 128, **bf), torch.zeros(128, 64, **bf))
    lay = layer(moe.Shape(64, 128, 8, 2, 2, 256), shared=sh)
    assert lay.stage_names() == ["route", "layout", "ffn", "shared", "combine"]
    assert lay.kernel_launches_per_step() == 1 + 1 + 1 + 1 + 3
