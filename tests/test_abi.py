"""The C ABI library loads on a host without a GPU and exports every entry point
that include/moe.h declares; its host-side argument checks answer without
touching the device."""
import ctypes
import dataclasses
import os
import re

import pytest

from combine_warp_top_gb300 import build as libbuild
from combine_warp_top_gb300 import moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return moe.load()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(moe_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_route", "moe_dispatch_layout", "moe_dispatch", "moe_expert_ffn",
                     "moe_combine", "moe_layer_forward", "moe_workspace_bytes", "moe_get_error",
                     "moe_status_str"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_host_side_checks_without_gpu(lib):
    shape = moe.Shape(4096, 7168, 256, 8, 8, 2048)
    assert moe.moe_workspace_bytes(shape) > 0
    assert moe.moe_workspace_bytes(moe.Shape(4096, 7168, 256, 8, 7, 2048)) == 0  # E % W
    assert moe.moe_workspace_bytes(moe.Shape(16, 8, 4, 5, 1, 8)) == 0           # k > E
    assert moe.moe_workspace_bytes(moe.Shape(16, 12, 4, 2, 1, 8)) == 0          # H % 8
    # a NULL logits pointer is refused before any CUDA call
    assert lib.moe_route(None, ctypes.byref(shape.c()), None, None, None) == 1
    assert lib.moe_dispatch(None, None, ctypes.byref(shape.c()), None, None) == 1
    assert lib.moe_get_error(None, None) == 3
    assert lib.moe_status_str(0) == b"ok"
    assert lib.moe_status_str(5) == b"device-side wait timed out"


def test_misaligned_rows_are_refused_without_gpu(lib):
    """A bf16 base address off the 16-byte grid (a view that starts one element
    into a tensor, say) is refused on the host, before any launch: the kernels
    move rows in 16-byte vectors."""
    shape = moe.Shape(64, 64, 8, 2, 2, 64)
    c = ctypes.byref(shape.c())
    fake = ctypes.c_void_p(0x10000)   # never dereferenced on the host
    odd = ctypes.c_void_p(0x10002)    # bf16 element 1 of a tensor at 0x10000
    lay = moe.MoeLayout(*([0x20000] * len(moe.LAYOUT_FIELDS)))
    L = ctypes.byref(lay)
    ws_bytes = ctypes.c_size_t(moe.moe_workspace_bytes(shape))
    assert lib.moe_dispatch(odd, L, c, fake, None) == 1
    assert lib.moe_dispatch(fake, L, c, odd, None) == 1
    assert lib.moe_combine(odd, fake, L, c, None, None, fake, None) == 1
    assert lib.moe_combine(fake, fake, L, c, None, odd, fake, None) == 1
    assert lib.moe_combine(fake, fake, L, c, None, None, odd, None) == 1
    assert lib.moe_ffn_gate_up(fake, L, c, fake, odd, fake, fake, ws_bytes, None) == 1
    assert lib.moe_ffn_down(odd, L, c, fake, fake, fake, ws_bytes, None) == 1
    assert lib.moe_ffn_gate_up_gather(odd, fake, ctypes.c_int64(64), L, c, fake, fake, fake,
                                      fake, ws_bytes, None) == 1


def test_binding_checks_sizes_against_the_shape(lib):
    """The C calls see only pointers, so the Python binding checks each tensor's
    element size and length against the shape before calling: an undersized
    or wrongly typed tensor, or a layout built for another shape, raises
    instead of sending a kernel out of bounds.  Each tensor is checked before
    its device check, so host tensors show it here for the first argument."""
    import torch
    shape = moe.Shape(64, 128, 8, 2, 2, 64)
    R, N, H, I, E = shape.R, shape.N, shape.H, shape.I, shape.E
    lay = moe.Layout.__new__(moe.Layout)  # host-side stand-in: no device arrays
    lay.shape = shape
    lay.c = moe.MoeLayout()
    bf = torch.bfloat16
    out = torch.empty(N * H, dtype=bf)
    with pytest.raises(ValueError, match="y: .* elements, the shape needs"):
        moe.moe_combine(torch.empty(R * H - 1, dtype=bf), torch.empty(R), lay, shape, None, None,
                        out)
    with pytest.raises(ValueError, match="y: expected 2-byte elements"):
        moe.moe_combine(torch.empty(R * H), torch.empty(R), lay, shape, None, None, out)
    with pytest.raises(ValueError, match="h: .* elements"):
        moe.moe_ffn_down(torch.empty(R * I - 8, dtype=bf), lay, shape,
                         torch.empty(E * H * I, dtype=bf), torch.empty(R * H, dtype=bf),
                         torch.empty(16, dtype=torch.uint8))
    with pytest.raises(ValueError, match="logits"):
        moe.moe_route(torch.empty(N * E - 1), shape, torch.empty(R, dtype=torch.int32),
                      torch.empty(R))
    # a layout must come from a shape with the same E, k, W and at least N tokens
    other = moe.Layout.__new__(moe.Layout)
    other.shape = moe.Shape(32, 128, 8, 2, 2, 64)
    with pytest.raises(ValueError, match="another shape"):
        moe._lay(other, shape)
    other.shape = moe.Shape(64, 128, 8, 2, 4, 64)
    with pytest.raises(ValueError, match="another shape"):
        moe._lay(other, shape)
    with pytest.raises(ValueError, match="another shape"):
        moe._lay(lay, moe.Shape(64, 128, 8, 2, 2, 64, dedup=True))
    moe._lay(lay, moe.Shape(16, 128, 8, 2, 2, 64))  # fewer tokens fit
    # correctly sized host tensors get as far as the device check
    with pytest.raises(ValueError, match="device tensors"):
        moe.moe_combine(torch.empty(R * H, dtype=bf), torch.empty(R), lay, shape, None, None,
                        out)


def test_workspace_grows_with_tokens(lib):
    small = moe.moe_workspace_bytes(moe.Shape(256, 64, 8, 2, 2, 64))
    large = moe.moe_workspace_bytes(moe.Shape(256 * 64, 64, 8, 2, 2, 64))
    assert large > small


def test_gemm_kernel_choice_is_an_argument(lib):
    """Which GEMM kernel runs is set by the shape's gemm field alone: values
    outside moe_gemm_kernel are refused, and whether the layer fuses its plain
    dispatch into the gate/up GEMM follows from the field (no environment or
    other global state is consulted)."""
    bad = moe.MoeShape(4096, 7168, 8, 2, 8, 2048, 0, 4)
    assert lib.moe_workspace_bytes(ctypes.byref(bad)) == 0
    assert lib.moe_route(None, ctypes.byref(bad), None, None, None) == 1
    # 8192 rows over 8 experts: the automatic choice is the CTA-pair kernel,
    # which has no gather mode, so the dispatch is not fused
    auto = moe.Shape(4096, 7168, 8, 2, 8, 2048)
    assert not moe.moe_layer_skips_dispatch(auto)
    assert moe.moe_layer_skips_dispatch(moe.Shape(4096, 7168, 8, 2, 8, 2048, gemm="single"))
    assert not moe.moe_layer_skips_dispatch(moe.Shape(4096, 7168, 8, 2, 8, 2048, gemm="pair"))
    # few rows per expert: the single-CTA kernel, dispatch fused, unless the pair is named
    few = moe.Shape(4096, 7168, 256, 8, 8, 2048)
    assert moe.moe_layer_skips_dispatch(few)
    assert not moe.moe_layer_skips_dispatch(moe.Shape(4096, 7168, 256, 8, 8, 2048, gemm="pair"))
    # the dedup form never skips the dispatch (its rows are the dedup rows)
    assert not moe.moe_layer_skips_dispatch(moe.Shape(4096, 7168, 256, 8, 8, 2048, dedup=True))
    with pytest.raises(ValueError):
        moe.Shape(64, 128, 8, 2, 2, 64, gemm="fast").c()


def test_fused_ffn_limits(lib):
    """The fused expert FFN (h on chip) takes H <= 256 only: its 128 x H fp32 y
    tile lives in TMEM next to the gate/up accumulators.  A shape that names
    it with a larger H is refused as unsupported by every call; with it the
    plain layer gathers its rows from x (no dispatch copy), the dedup layer
    does not."""
    assert moe.GEMM_KERNELS["fused"] == 3
    for H in (8, 128, 200, 256):
        s = moe.Shape(300, H, 8, 2, 4, 384, gemm="fused")
        assert moe.moe_ffn_fused_supported(s)
        assert moe.moe_workspace_bytes(s) > 0
        assert moe.moe_layer_skips_dispatch(s)
        assert not moe.moe_layer_skips_dispatch(dataclasses.replace(s, dedup=True))
        # I is not limited
        assert moe.moe_ffn_fused_supported(moe.Shape(300, H, 8, 2, 4, 14336))
    # the layer fuses its FFN when the shape names the fused kernel, and by
    # default for H <= 256 (plain form; dedup: H <= 128); then it gathers
    # plain rows from x itself, whichever kernel the separate GEMM calls would run
    for gemm, H, want in (("auto", 128, True), ("auto", 8, True), ("auto", 136, True),
                          ("auto", 256, True), ("fused", 256, True), ("auto", 264, False),
                          ("auto", 7168, False), ("fused", 200, True), ("single", 128, False),
                          ("pair", 128, False)):
        s = moe.Shape(16384, H, 16, 4, 4, 1408, gemm=gemm)
        assert moe.moe_layer_fuses_ffn(s) == want, (gemm, H)
        assert moe.moe_layer_skips_dispatch(s) == (want or gemm == "single")
    assert not moe.moe_layer_fuses_ffn(moe.Shape(64, 264, 8, 2, 2, 64, gemm="fused"))
    # few rows and a long I: the two GEMMs (which spread over I); a short I fuses
    assert not moe.moe_layer_fuses_ffn(moe.Shape(200, 128, 16, 4, 4, 512))
    assert moe.moe_layer_fuses_ffn(moe.Shape(64, 128, 8, 2, 2, 256))
    assert moe.moe_layer_fuses_ffn(moe.Shape(1024, 128, 16, 4, 4, 512))
    # dedup layers fuse by default only up to H = 128
    assert moe.moe_layer_fuses_ffn(moe.Shape(4096, 128, 8, 2, 4, 384, dedup=True))
    assert not moe.moe_layer_fuses_ffn(moe.Shape(4096, 136, 8, 2, 4, 384, dedup=True))
    assert moe.moe_layer_fuses_ffn(moe.Shape(300, 256, 8, 2, 4, 384, dedup=True, gemm="fused"))
    wide = moe.Shape(300, 264, 8, 2, 4, 384, gemm="fused")
    assert moe.moe_workspace_bytes(wide) == 0
    assert lib.moe_route(None, ctypes.byref(wide.c()), None, None, None) == 2
    assert not moe.moe_ffn_fused_supported(moe.Shape(300, 264, 8, 2, 4, 384))
    assert not moe.moe_ffn_fused_supported(moe.Shape(4096, 7168, 256, 8, 8, 2048))
    # refused on the host before anything is launched
    s = moe.Shape(64, 128, 8, 2, 2, 64)
    lay = moe.MoeLayout()
    ws = ctypes.create_string_buffer(moe.moe_workspace_bytes(s))
    big = moe.Shape(64, 264, 8, 2, 2, 64)
    assert lib.moe_ffn_fused(None, None, 64, ctypes.byref(lay), ctypes.byref(big.c()), None, None,
                             None, None, ws, len(ws), None) == 1  # empty layout first
    assert lib.moe_ffn_fused(None, None, 64, None, ctypes.byref(s.c()), None, None, None, None,
                             ws, len(ws), None) == 1


def test_weight_layout_field_and_packed_sizes(lib):
    """shape.weights takes the moe_weight_layout values only; the packed sizes
    are the block counts of the header's definition (gate/up: E * ceil(I/128)
    * ceil(H/64) blocks, down: E * ceil(H/256) * ceil(I/64) blocks, 32 KB
    each), whatever the field says; the packed calls accept w_up = NULL."""
    bad = moe.MoeShape(300, 256, 8, 2, 4, 384, 0, 0, 2)
    assert lib.moe_workspace_bytes(ctypes.byref(bad)) == 0
    for weights in ("row_major", "packed"):
        s = moe.Shape(300, 256, 8, 2, 4, 384, weights=weights)
        assert moe.moe_workspace_bytes(s) > 0
        assert moe.moe_packed_gate_up_bytes(s) == 8 * 3 * 4 * 32768
        assert moe.moe_packed_down_bytes(s) == 8 * 1 * 6 * 32768
    s = moe.Shape(4096, 7168, 256, 8, 8, 2048)
    assert moe.moe_packed_gate_up_bytes(s) == 2 * 256 * 2048 * 7168 * 2  # no padding
    assert moe.moe_packed_down_bytes(s) == 256 * 7168 * 2048 * 2
    with pytest.raises(ValueError):
        moe.Shape(64, 128, 8, 2, 2, 64, weights="tiled").c()
    # packed weights of 2^31 rows of 64 bf16 or more are refused (32-bit TMA rows)
    huge = moe.Shape(16, 65536, 1024, 2, 1, 65536, weights="packed")
    assert moe.moe_workspace_bytes(huge) == 0
    # a packed call needs no w_up: refused on the missing rows pointer, not on w_up
    ok = moe.Shape(64, 128, 8, 2, 2, 64, weights="packed")
    st = lib.moe_ffn_gate_up(None, None, ctypes.byref(ok.c()), None, None, None, None, 0, None)
    assert st == 1


def test_library_sources_read_no_environment():
    csrc = os.path.join(ROOT, "combine_warp_top_gb300", "csrc")
    for fn in os.listdir(csrc):
        text = open(os.path.join(csrc, fn)).read()
        assert "getenv" not in text, fn
