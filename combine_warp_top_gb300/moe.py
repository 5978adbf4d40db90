"""Python binding of libmoe (include/moe.h): argument marshalling only.

Every function below has the name of the C entry point it calls and takes
torch CUDA tensors in place of device pointers.  All arithmetic runs in the
library's kernels; if libmoe.so cannot be loaded the binding raises -- there
is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

SHAPE_FIELDS = ("N", "H", "E", "k", "W", "I", "dedup", "gemm", "weights")
# moe_gemm_kernel values of include/moe.h
GEMM_KERNELS = {"auto": 0, "single": 1, "pair": 2, "fused": 3}
# moe_weight_layout values of include/moe.h
WEIGHT_LAYOUTS = {"row_major": 0, "packed": 1}
LAYOUT_FIELDS = ("expert_counts", "expert_offsets", "rank_offsets", "row_token", "pair_row",
                 "dedup_counts", "dedup_offsets", "dedup_row_token", "pair_dedup_row",
                 "expand_src", "n_dedup_rows")
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_DEVICE_ASSERT"}


class MoeShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in SHAPE_FIELDS]


class MoeLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in LAYOUT_FIELDS]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({_lib_status_str(status)})")


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmoe.so (built by __graft_entry__.build()).  Raises if missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libmoe.so not built at {path}; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, S, I32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    shp, lay = ctypes.POINTER(MoeShape), ctypes.POINTER(MoeLayout)
    sigs = {
        "moe_workspace_bytes": (S, [shp]),
        "moe_packed_gate_up_bytes": (S, [shp]),
        "moe_packed_down_bytes": (S, [shp]),
        "moe_pack_weights": (I32, [P, P, P, shp, P, P, P]),
        "moe_route": (I32, [P, shp, P, P, P]),
        "moe_route_full_softmax": (I32, [P, shp, P, P, P]),
        "moe_route_sigmoid_bias": (I32, [P, P, shp, P, P, P]),
        "moe_dispatch_layout": (I32, [P, P, shp, lay, P, S, P]),
        "moe_dispatch": (I32, [P, lay, shp, P, P]),
        "moe_expert_ffn": (I32, [P, lay, shp, P, P, P, P, P, P, P, S, P]),
        "moe_expand": (I32, [P, lay, shp, P, P]),
        "moe_ffn_gate_up": (I32, [P, lay, shp, P, P, P, P, S, P]),
        "moe_ffn_down": (I32, [P, lay, shp, P, P, P, S, P]),
        "moe_ffn_gate_up_gather": (I32, [P, P, ctypes.c_int64, lay, shp, P, P, P, P, S, P]),
        "moe_ffn_fused": (I32, [P, P, ctypes.c_int64, lay, shp, P, P, P, P, P, S, P]),
        "moe_ffn_fused_supported": (ctypes.c_int32, [shp]),
        "moe_combine": (I32, [P, P, lay, shp, P, P, P, P]),
        "moe_ffn_down_combine": (I32, [P, P, lay, shp, P, P, P, P, P, S, P]),
        "moe_layer_forward": (I32, [P, P, P, P, P, P, P, shp, P, P, lay, P, P, P, P, P, P, P, S,
                                    P]),
        "moe_dispatch_layout_noalloc": (I32, [P, P, shp, lay, P]),
        "moe_layer_skips_dispatch": (ctypes.c_int32, [shp]),
        "moe_layer_fuses_ffn": (ctypes.c_int32, [shp]),
        "moe_coselection": (I32, [P, shp, P, P, S, P]),
        "moe_shared_expert_ffn": (I32, [P, shp, ctypes.c_int32, P, P, P, P, P, P, S, P]),
        "moe_combine_shared": (I32, [P, P, lay, shp, P, P, P, P, P]),
        "moe_placement_search": (I32, [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_int64, P, P]),
        "moe_selftest_wait_timeout": (I32, [P, ctypes.c_int64, P]),
        "moe_get_error": (I32, [P, P]),
        "moe_status_str": (ctypes.c_char_p, [I32]),
    }
    for name, (res, args) in sigs.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _lib_status_str(status: int) -> str:
    try:
        return load().moe_status_str(int(status)).decode()
    except Exception:
        return "?"


def _check(status: int, where: str):
    if status != 0:
        raise MoeError(status, where)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("libmoe takes device tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _sized(t, count, esize, what):
    """Pointer of t after checking that it holds at least `count` elements of
    `esize` bytes: what the C call reads or writes for its shape.  The C ABI
    sees only pointers, so a smaller tensor would send the kernels out of
    bounds.  None passes (the C call decides whether NULL is allowed)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what}: expected a torch tensor")
    if t.element_size() != esize:
        raise ValueError(f"{what}: expected {esize}-byte elements, got {t.dtype}")
    if t.numel() < count:
        raise ValueError(f"{what}: {t.numel()} elements, the shape needs {count}")
    return _ptr(t)


def _bf16(t, count, what):
    return _sized(t, count, 2, what)


def _i32(t, count, what):
    return _sized(t, count, 4, what)


def _f32(t, count, what):
    return _sized(t, count, 4, what)


def _ws(ws):
    """(pointer, size in bytes) of a workspace tensor of any dtype."""
    return _ptr(ws), ws.numel() * ws.element_size()


def _lay(layout, shape):
    """The C struct of a layout built for this shape's E, k and W, for at least
    its N tokens, with the dedup arrays if the shape deduplicates."""
    ls = layout.shape
    if (ls.E, ls.k, ls.W) != (shape.E, shape.k, shape.W) or ls.N < shape.N or \
            (shape.dedup and not ls.dedup):
        raise ValueError("the layout was built for another shape")
    return ctypes.byref(layout.c)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ---- shapes, layouts, buffers ----------------------------------------------------------

@dataclass(frozen=True)
class Shape:
    N: int
    H: int
    E: int
    k: int
    W: int
    I: int
    dedup: bool = False
    # which grouped-GEMM kernel runs: "auto", "single" (128-row tiles, one CTA),
    # "pair" (256-row tiles on a 2-CTA cluster) or "fused" (the whole expert
    # FFN in one kernel with h on chip, H <= 256); see moe_gemm_kernel
    gemm: str = "auto"
    # layout of the expert weights the calls take: "row_major" (nn.Linear) or
    # "packed" (moe_pack_weights); see moe_weight_layout
    weights: str = "row_major"

    def c(self) -> MoeShape:
        if self.gemm not in GEMM_KERNELS:
            raise ValueError(f"gemm must be one of {sorted(GEMM_KERNELS)}")
        if self.weights not in WEIGHT_LAYOUTS:
            raise ValueError(f"weights must be one of {sorted(WEIGHT_LAYOUTS)}")
        return MoeShape(self.N, self.H, self.E, self.k, self.W, self.I, int(bool(self.dedup)),
                        GEMM_KERNELS[self.gemm], WEIGHT_LAYOUTS[self.weights])

    @property
    def R(self) -> int:
        return self.N * self.k

    @property
    def R_d_max(self) -> int:
        return self.N * min(self.k, self.W)


class Layout:
    """Device arrays of one dispatch layout (see moe_layout in include/moe.h)."""

    def __init__(self, shape: Shape, device="cuda"):
        self.shape = shape
        N, E, k, W = shape.N, shape.E, shape.k, shape.W
        i32 = dict(dtype=torch.int32, device=device)
        sizes = dict(expert_counts=E, expert_offsets=E + 1, rank_offsets=W + 1,
                     row_token=N * k, pair_row=N * k)
        if shape.dedup:
            sizes.update(dedup_counts=W, dedup_offsets=W + 1, dedup_row_token=N * min(k, W),
                         pair_dedup_row=N * k, expand_src=N * k, n_dedup_rows=1)
        self.tensors = {n: torch.zeros(max(s, 1), **i32) for n, s in sizes.items()}
        self.c = MoeLayout(*[ctypes.c_void_p(self.tensors[n].data_ptr()) if n in self.tensors
                             else None for n in LAYOUT_FIELDS])

    def __getitem__(self, name):
        return self.tensors[name]


def moe_workspace_bytes(shape: Shape) -> int:
    return int(load().moe_workspace_bytes(ctypes.byref(shape.c())))


def workspace(shape: Shape, device="cuda") -> torch.Tensor:
    n = moe_workspace_bytes(shape)
    if n == 0:
        raise MoeError(1, "moe_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


# ---- the C entry points ----------------------------------------------------------------
# Each wrapper checks its tensors' element sizes and lengths against the shape
# (the C side cannot), then passes plain pointers.

def _rows_d(shape: Shape) -> int:
    return shape.R_d_max if shape.dedup else shape.R


def moe_packed_gate_up_bytes(shape: Shape) -> int:
    return int(load().moe_packed_gate_up_bytes(ctypes.byref(shape.c())))


def moe_packed_down_bytes(shape: Shape) -> int:
    return int(load().moe_packed_down_bytes(ctypes.byref(shape.c())))


def _gate_up_w(shape: Shape, w_gate, w_up):
    """Pointers of the gate/up weights in the shape's layout (packed: both in
    w_gate, w_up not read and may be None)."""
    s = shape
    if s.weights == "packed":
        return (_bf16(w_gate, moe_packed_gate_up_bytes(s) // 2, "w_gate (packed gate/up)"),
                _bf16(w_up, 0, "w_up"))
    return (_bf16(w_gate, s.E * s.I * s.H, "w_gate"), _bf16(w_up, s.E * s.I * s.H, "w_up"))


def _down_w(shape: Shape, w_down):
    s = shape
    if s.weights == "packed":
        return _bf16(w_down, moe_packed_down_bytes(s) // 2, "w_down (packed)")
    return _bf16(w_down, s.E * s.H * s.I, "w_down")


def moe_pack_weights(w_gate, w_up, w_down, shape: Shape, gate_up_packed, down_packed,
                     stream=None):
    """Row-major weights -> the packed layout (either output may be None)."""
    s = dataclasses.replace(shape, weights="row_major")
    gu = down = None
    if gate_up_packed is not None:
        gu = _bf16(gate_up_packed, moe_packed_gate_up_bytes(s) // 2, "gate_up_packed")
        w_gate = _bf16(w_gate, s.E * s.I * s.H, "w_gate")
        w_up = _bf16(w_up, s.E * s.I * s.H, "w_up")
    else:
        w_gate = w_up = None
    if down_packed is not None:
        down = _bf16(down_packed, moe_packed_down_bytes(s) // 2, "down_packed")
        w_down = _bf16(w_down, s.E * s.H * s.I, "w_down")
    else:
        w_down = None
    _check(load().moe_pack_weights(w_gate, w_up, w_down, ctypes.byref(s.c()), gu, down,
                                   _stream(stream)), "moe_pack_weights")


def pack_weights(shape: Shape, w_gate, w_up, w_down, stream=None):
    """Allocates and fills the packed gate/up and down weights of `shape`;
    returns (gate_up_packed, down_packed), flat bf16 device tensors."""
    s = dataclasses.replace(shape, weights="row_major")
    dev = w_gate.device
    gu = torch.empty(moe_packed_gate_up_bytes(s) // 2, dtype=torch.bfloat16, device=dev)
    dn = torch.empty(moe_packed_down_bytes(s) // 2, dtype=torch.bfloat16, device=dev)
    moe_pack_weights(w_gate, w_up, w_down, s, gu, dn, stream)
    return gu, dn


def moe_route(logits, shape: Shape, topk_ids, topk_w, stream=None):
    s = shape
    _check(load().moe_route(_f32(logits, s.N * s.E, "logits"), ctypes.byref(s.c()),
                            _i32(topk_ids, s.R, "topk_ids"), _f32(topk_w, s.R, "topk_w"),
                            _stream(stream)), "moe_route")


def moe_route_full_softmax(logits, shape: Shape, topk_ids, topk_w, stream=None):
    s = shape
    _check(load().moe_route_full_softmax(_f32(logits, s.N * s.E, "logits"), ctypes.byref(s.c()),
                                         _i32(topk_ids, s.R, "topk_ids"),
                                         _f32(topk_w, s.R, "topk_w"), _stream(stream)),
           "moe_route_full_softmax")


def moe_route_sigmoid_bias(logits, bias, shape: Shape, topk_ids, topk_w, stream=None):
    s = shape
    _check(load().moe_route_sigmoid_bias(_f32(logits, s.N * s.E, "logits"),
                                         _f32(bias, s.E, "bias"), ctypes.byref(s.c()),
                                         _i32(topk_ids, s.R, "topk_ids"),
                                         _f32(topk_w, s.R, "topk_w"), _stream(stream)),
           "moe_route_sigmoid_bias")


def moe_dispatch_layout(topk_ids, placement, shape: Shape, layout: Layout, ws, stream=None):
    s = shape
    _check(load().moe_dispatch_layout(_i32(topk_ids, s.R, "topk_ids"),
                                      _i32(placement, s.E, "placement"), ctypes.byref(s.c()),
                                      _lay(layout, s), *_ws(ws), _stream(stream)),
           "moe_dispatch_layout")


def moe_dispatch_layout_noalloc(topk_ids, placement, shape: Shape, layout: Layout, stream=None):
    s = shape
    _check(load().moe_dispatch_layout_noalloc(_i32(topk_ids, s.R, "topk_ids"),
                                              _i32(placement, s.E, "placement"),
                                              ctypes.byref(s.c()), _lay(layout, s),
                                              _stream(stream)), "moe_dispatch_layout_noalloc")


def moe_dispatch(x, layout: Layout, shape: Shape, xd, stream=None):
    s = shape
    _check(load().moe_dispatch(_bf16(x, s.N * s.H, "x"), _lay(layout, s), ctypes.byref(s.c()),
                               _bf16(xd, _rows_d(s) * s.H, "xd"), _stream(stream)),
           "moe_dispatch")


def moe_expert_ffn(xd, layout: Layout, shape: Shape, w_gate, w_up, w_down, xe, h, y, ws,
                   stream=None):
    s = shape
    _check(load().moe_expert_ffn(_bf16(xd, _rows_d(s) * s.H, "xd"), _lay(layout, s),
                                 ctypes.byref(s.c()), *_gate_up_w(s, w_gate, w_up),
                                 _down_w(s, w_down), _ptr(xe),
                                 _bf16(h, s.R * s.I, "h"), _bf16(y, s.R * s.H, "y"), *_ws(ws),
                                 _stream(stream)), "moe_expert_ffn")


def moe_expand(xd, layout: Layout, shape: Shape, xe, stream=None):
    s = shape
    _check(load().moe_expand(_bf16(xd, s.R_d_max * s.H, "xd"), _lay(layout, s),
                             ctypes.byref(s.c()), _bf16(xe, s.R * s.H, "xe"), _stream(stream)),
           "moe_expand")


def moe_ffn_gate_up(rows, layout: Layout, shape: Shape, w_gate, w_up, h, ws, stream=None):
    s = shape
    _check(load().moe_ffn_gate_up(_bf16(rows, s.R * s.H, "rows"), _lay(layout, s),
                                  ctypes.byref(s.c()), *_gate_up_w(s, w_gate, w_up),
                                  _bf16(h, s.R * s.I, "h"),
                                  *_ws(ws), _stream(stream)), "moe_ffn_gate_up")


def moe_ffn_gate_up_gather(src, row_index, layout: Layout, shape: Shape, w_gate, w_up, h, ws,
                           stream=None):
    """src: the [src_rows, H] rows that row_index points into."""
    s = shape
    src_rows = src.numel() // s.H
    _check(load().moe_ffn_gate_up_gather(_bf16(src, src_rows * s.H, "src"),
                                         _i32(row_index, s.R, "row_index"), src_rows,
                                         _lay(layout, s), ctypes.byref(s.c()),
                                         *_gate_up_w(s, w_gate, w_up),
                                         _bf16(h, s.R * s.I, "h"), *_ws(ws), _stream(stream)),
           "moe_ffn_gate_up_gather")


def moe_ffn_fused(src, row_index, layout: Layout, shape: Shape, w_gate, w_up, w_down, y, ws,
                  stream=None):
    """The expert FFN with h kept on chip: y for the problem's rows, row i
    being src[row_index[i]] (row_index None: src[i]); src is [src_rows, H]."""
    s = shape
    src_rows = src.numel() // s.H
    _check(load().moe_ffn_fused(_bf16(src, src_rows * s.H, "src"),
                                _i32(row_index, s.R, "row_index"), src_rows, _lay(layout, s),
                                ctypes.byref(s.c()), *_gate_up_w(s, w_gate, w_up),
                                _down_w(s, w_down), _bf16(y, s.R * s.H, "y"), *_ws(ws),
                                _stream(stream)), "moe_ffn_fused")


def moe_ffn_fused_supported(shape: Shape) -> bool:
    return bool(load().moe_ffn_fused_supported(ctypes.byref(shape.c())))


def moe_ffn_down_combine(h, topk_w, layout: Layout, shape: Shape, w_down, residual, acc, out,
                         ws, stream=None):
    s = shape
    _check(load().moe_ffn_down_combine(_bf16(h, s.R * s.I, "h"), _f32(topk_w, s.R, "topk_w"),
                                       _lay(layout, s), ctypes.byref(s.c()), _down_w(s, w_down),
                                       _bf16(residual, s.N * s.H, "residual"),
                                       _f32(acc, s.N * s.H, "acc"), _bf16(out, s.N * s.H, "out"),
                                       *_ws(ws), _stream(stream)), "moe_ffn_down_combine")


def moe_layer_skips_dispatch(shape: Shape) -> bool:
    """True when the layer gathers its plain rows inside the gate/up GEMM
    (no moe_dispatch copy) for this shape."""
    return bool(load().moe_layer_skips_dispatch(ctypes.byref(shape.c())))


def moe_layer_fuses_ffn(shape: Shape) -> bool:
    """True when the layer runs its expert FFN as the one fused kernel
    (moe_ffn_fused, h kept on chip) for this shape."""
    return bool(load().moe_layer_fuses_ffn(ctypes.byref(shape.c())))


def moe_ffn_down(h, layout: Layout, shape: Shape, w_down, y, ws, stream=None):
    s = shape
    _check(load().moe_ffn_down(_bf16(h, s.R * s.I, "h"), _lay(layout, s), ctypes.byref(s.c()),
                               _down_w(s, w_down), _bf16(y, s.R * s.H, "y"), *_ws(ws),
                               _stream(stream)),
           "moe_ffn_down")


def moe_combine(y, topk_w, layout: Layout, shape: Shape, partial, residual, out, stream=None):
    s = shape
    _check(load().moe_combine(_bf16(y, s.R * s.H, "y"), _f32(topk_w, s.R, "topk_w"),
                              _lay(layout, s), ctypes.byref(s.c()),
                              _bf16(partial, s.R_d_max * s.H, "partial"),
                              _bf16(residual, s.N * s.H, "residual"),
                              _bf16(out, s.N * s.H, "out"), _stream(stream)), "moe_combine")


def moe_layer_forward(logits, x, placement, w_gate, w_up, w_down, residual, shape: Shape,
                      topk_ids, topk_w, layout: Layout, xd, xe, h, y, partial, out, ws,
                      stream=None):
    s = shape
    # xd is not written when the dispatch is fused into the gate/up GEMM
    xd_rows = 0 if moe_layer_skips_dispatch(s) else _rows_d(s)
    _check(load().moe_layer_forward(
        _f32(logits, s.N * s.E, "logits"), _bf16(x, s.N * s.H, "x"),
        _i32(placement, s.E, "placement"), *_gate_up_w(s, w_gate, w_up), _down_w(s, w_down),
        _bf16(residual, s.N * s.H, "residual"), ctypes.byref(s.c()),
        _i32(topk_ids, s.R, "topk_ids"), _f32(topk_w, s.R, "topk_w"), _lay(layout, s),
        _bf16(xd, xd_rows * s.H, "xd"), _ptr(xe), _bf16(h, s.R * s.I, "h"),
        _bf16(y, s.R * s.H, "y"), _bf16(partial, s.R_d_max * s.H, "partial"),
        _bf16(out, s.N * s.H, "out"), *_ws(ws), _stream(stream)), "moe_layer_forward")


def moe_shared_expert_ffn(x, shape: Shape, I_shared: int, w_gate_s, w_up_s, w_down_s, h_s, y_s, ws,
                          stream=None):
    s, Is = shape, I_shared
    _check(load().moe_shared_expert_ffn(_bf16(x, s.N * s.H, "x"), ctypes.byref(s.c()), Is,
                                        _bf16(w_gate_s, Is * s.H, "w_gate_s"),
                                        _bf16(w_up_s, Is * s.H, "w_up_s"),
                                        _bf16(w_down_s, s.H * Is, "w_down_s"),
                                        _bf16(h_s, s.N * Is, "h_s"), _bf16(y_s, s.N * s.H, "y_s"),
                                        *_ws(ws), _stream(stream)), "moe_shared_expert_ffn")


def moe_combine_shared(y, topk_w, layout: Layout, shape: Shape, partial, y_shared, residual, out,
                       stream=None):
    s = shape
    _check(load().moe_combine_shared(_bf16(y, s.R * s.H, "y"), _f32(topk_w, s.R, "topk_w"),
                                     _lay(layout, s), ctypes.byref(s.c()),
                                     _bf16(partial, s.R_d_max * s.H, "partial"),
                                     _bf16(y_shared, s.N * s.H, "y_shared"),
                                     _bf16(residual, s.N * s.H, "residual"),
                                     _bf16(out, s.N * s.H, "out"), _stream(stream)),
           "moe_combine_shared")


def moe_coselection(topk_ids, shape: Shape, coselect, ws, stream=None):
    s = shape
    _check(load().moe_coselection(_i32(topk_ids, s.R, "topk_ids"), ctypes.byref(s.c()),
                                  _i32(coselect, s.E * s.E, "coselect"), *_ws(ws),
                                  _stream(stream)), "moe_coselection")


def moe_placement_search(coselect_host, ranks: int, nodes: int = 1, max_swaps: int = 1 << 20):
    """Host call: coselect_host is a CPU int32 tensor [E, E]; returns
    (placement int32 CPU tensor [E], number of swaps)."""
    if coselect_host.is_cuda or coselect_host.dtype != torch.int32:
        raise ValueError("coselect must be a CPU int32 tensor")
    c = coselect_host.contiguous()
    E = c.shape[0]
    placement = torch.empty(E, dtype=torch.int32)
    swaps = ctypes.c_int64(0)
    _check(load().moe_placement_search(ctypes.c_void_p(c.data_ptr()), E, ranks, nodes, max_swaps,
                                       ctypes.c_void_p(placement.data_ptr()), ctypes.byref(swaps)),
           "moe_placement_search")
    return placement, int(swaps.value)


def moe_selftest_wait_timeout(ws, limit_cycles: int, stream=None):
    _check(load().moe_selftest_wait_timeout(_ptr(ws), limit_cycles, _stream(stream)),
           "moe_selftest_wait_timeout")


def moe_get_error(ws, stream=None) -> int:
    return int(load().moe_get_error(_ptr(ws), _stream(stream)))


def moe_status_str(status: int) -> str:
    return _lib_status_str(status)


def layout_launches(shape: Shape) -> int:
    """Kernels moe_dispatch_layout launches for this shape: count and scatter,
    plus a separate scan when the per-block count tables (one int32 per block
    of 256 tokens and slot, and per block and rank with dedup, each rounded
    up to 16 bytes) exceed the 64 KB that each scatter block scans itself
    (csrc/layout.cu, kScanTableBytes; workspaces from this module are
    256-byte aligned, as the in-shared-memory scan needs); the scatter alone
    when one block of 256 tokens holds them all."""
    nb = (shape.N + 255) // 256
    if nb <= 1:
        return 1
    pad4 = lambda n: (n + 3) // 4 * 4  # noqa: E731
    table = 4 * (pad4(nb * shape.E) + (pad4(nb * shape.W) if shape.dedup else 0))
    return 2 if table <= 64 * 1024 else 3


# ---- a layer with its buffers ----------------------------------------------------------

class MoELayer:
    """Owns the device buffers of one layer shape (all allocated by torch) and
    runs moe_layer_forward on them.  Weights are bf16 tensors [E, I, H] (gate,
    up) and [E, H, I] (down) when shape.weights is "row_major", or the packed
    tensors of pack_weights (w_up None) when it is "packed"; placement int32
    [E] or None."""

    def __init__(self, shape: Shape, w_gate, w_up, w_down, placement=None, device="cuda",
                 shared=None, fuse_combine=False, pack=True):
        """shared: optional (w_gate_s [I_s, H], w_up_s [I_s, H], w_down_s [H, I_s])
        of a shared expert run on every token.  fuse_combine: run the down GEMM
        with the combine in its epilogue (moe_ffn_down_combine, fp32
        accumulator) instead of moe_ffn_down + moe_combine.  pack: copy
        row-major weights once into the packed layout (moe_pack_weights) and
        run the layer on that copy (the layer's shape becomes "packed"); the
        results are bit-identical, the weight stream faster."""
        if fuse_combine and shared is not None:
            raise ValueError("the combine fused into the down GEMM adds no shared expert")
        if fuse_combine and shape.gemm == "fused":
            raise ValueError("the fused expert FFN has no down GEMM to put the combine in")
        if pack and shape.weights == "row_major":
            w_gate, w_down = pack_weights(shape, w_gate, w_up, w_down)
            w_up = None
            shape = dataclasses.replace(shape, weights="packed")
        self.shape = shape
        self.fuse_combine = fuse_combine
        self.w_gate, self.w_up, self.w_down = w_gate, w_up, w_down
        self.placement = placement
        self.shared = shared
        if shared is not None:
            I_s = shared[0].shape[0]
            self.I_shared = I_s
            self.h_s = torch.empty(max(shape.N, 1), I_s, dtype=torch.bfloat16, device=device)
            self.y_s = torch.empty(max(shape.N, 1), shape.H, dtype=torch.bfloat16, device=device)
        N, H, I, k = shape.N, shape.H, shape.I, shape.k
        bf = dict(dtype=torch.bfloat16, device=device)
        self.topk_ids = torch.empty(max(N * k, 1), dtype=torch.int32, device=device)
        self.topk_w = torch.empty(max(N * k, 1), dtype=torch.float32, device=device)
        self.layout = Layout(shape, device)
        rows_d = shape.R_d_max if shape.dedup else shape.R
        # plain rows gathered inside the gate/up GEMM need no dispatch buffer
        self.fused_dispatch = moe_layer_skips_dispatch(shape)
        # the expert FFN as one kernel (h on chip), unless the combine is to go
        # into the down GEMM's epilogue
        self.fused_ffn = moe_layer_fuses_ffn(shape) and not fuse_combine
        self.xd = torch.empty(1 if self.fused_dispatch else max(rows_d, 1), H, **bf)
        self.xe = None  # the dedup expansion happens inside the gate/up GEMM
        self.h = torch.empty(max(shape.R, 1), I, **bf)
        self.y = torch.empty(max(shape.R, 1), H, **bf)
        # the dedup combine keeps its partial rows in registers (moe_combine with
        # partial = NULL); a caller who wants them written passes its own buffer
        self.partial = None
        self.out = torch.empty(max(N, 1), H, **bf)
        self.acc = (torch.empty(max(N, 1), H, dtype=torch.float32, device=device)
                    if fuse_combine else None)
        self.ws = workspace(shape, device)

    def forward(self, logits, x, residual=None, out=None, stream=None):
        out = self.out if out is None else out
        if self.shared is not None or self.fuse_combine:
            return self.forward_stages(logits, x, residual, out, stream)
        moe_layer_forward(logits, x, self.placement, self.w_gate, self.w_up, self.w_down,
                          residual, self.shape, self.topk_ids, self.topk_w, self.layout,
                          self.xd, self.xe, self.h, self.y, self.partial, out, self.ws, stream)
        return out

    def capture(self, logits, x, residual=None, out=None):
        """Capture one forward on these exact buffers into a CUDA graph and
        return it; graph.replay() then reruns the whole layer (all of its
        kernel launches) on whatever the buffers hold, with one launch of the
        graph.  The first forward (outside the capture) sets the kernels'
        shared-memory attributes."""
        out = self.out if out is None else out
        self.forward(logits, x, residual, out)  # warm-up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.forward(logits, x, residual, out)
        return g

    STAGES = ("route", "layout", "dispatch", "gate_up", "ffn", "down", "shared", "combine",
              "down_combine")

    def stage_names(self):
        """The stages forward_stages() runs for this layer, in order: no
        separate dispatch when the gate/up GEMM gathers the plain rows from x,
        no shared expert unless one is set."""
        fused = ("down_combine",) if self.fuse_combine else ("down", "combine")
        # fused FFN: one "ffn" stage (moe_ffn_fused) instead of gate_up + down
        ffn = ("ffn",) if self.fused_ffn else ("gate_up", "down")
        return [n for n in self.STAGES
                if (n != "dispatch" or not self.fused_dispatch)
                and (n != "shared" or self.shared is not None)
                and (n not in ("down", "combine", "down_combine") or n in fused)
                and (n not in ("gate_up", "ffn", "down") or n in ffn)]

    def forward_stages(self, logits, x, residual=None, out=None, stream=None, events=None):
        """The same kernels as forward(), one C call per stage of the pages'
        pipeline.  If ``events`` maps stage names to (start, end) CUDA events,
        they are recorded around each stage on the stream."""
        out = self.out if out is None else out
        st = torch.cuda.current_stream() if stream is None else stream
        for name in self.stage_names():
            if events is not None and name in events:
                events[name][0].record(st)
            self.run_stage(name, logits, x, residual, out, st)
            if events is not None and name in events:
                events[name][1].record(st)
        return out

    def run_stage(self, name, logits, x, residual, out, st):
        """One stage of forward_stages() on this layer's buffers (one C call)."""
        s = self.shape
        if name == "route":
            moe_route(logits, s, self.topk_ids, self.topk_w, st)
        elif name == "layout":
            moe_dispatch_layout(self.topk_ids, self.placement, s, self.layout, self.ws, st)
        elif name == "dispatch":
            moe_dispatch(x, self.layout, s, self.xd, st)
        elif name == "gate_up":
            self._gate_up(x, st)
        elif name == "ffn":
            self._ffn_fused(x, st)
        elif name == "down_combine":
            moe_ffn_down_combine(self.h, self.topk_w, self.layout, s, self.w_down, residual,
                                 self.acc, out, self.ws, st)
        elif name == "down":
            moe_ffn_down(self.h, self.layout, s, self.w_down, self.y, self.ws, st)
        elif name == "shared":
            moe_shared_expert_ffn(x, s, self.I_shared, *self.shared, self.h_s, self.y_s, self.ws, st)
        elif name == "combine":
            if self.shared is not None:
                moe_combine_shared(self.y, self.topk_w, self.layout, s, self.partial, self.y_s,
                                   residual, out, st)
            else:
                moe_combine(self.y, self.topk_w, self.layout, s, self.partial, residual, out, st)
        else:
            raise ValueError(f"unknown stage {name}")

    def _ffn_fused(self, x, st):
        """The expert FFN as moe_layer_forward runs it when it fuses the FFN:
        one kernel, rows gathered like the gate/up stage's (dedup rows through
        expand_src, plain rows of x through row_token)."""
        s, lay = self.shape, self.layout
        if s.dedup:
            src, index = self.xd, lay["expand_src"]
        elif self.fused_dispatch:
            src, index = x, lay["row_token"]
        else:
            src, index = self.xd, None
        moe_ffn_fused(src, index, lay, s, self.w_gate, self.w_up, self.w_down, self.y, self.ws, st)

    def _gate_up(self, x, st):
        """The gate/up stage as moe_layer_forward runs it: dedup rows expanded
        by the GEMM's gather warps; plain rows gathered from x when the
        dispatch is fused, else read from the dispatched rows."""
        s, lay = self.shape, self.layout
        if s.dedup:
            moe_ffn_gate_up_gather(self.xd, lay["expand_src"], lay, s, self.w_gate, self.w_up,
                                   self.h, self.ws, st)
        elif self.fused_dispatch:
            moe_ffn_gate_up_gather(x, lay["row_token"], lay, s, self.w_gate, self.w_up, self.h,
                                   self.ws, st)
        else:
            moe_ffn_gate_up(self.xd, lay, s, self.w_gate, self.w_up, self.h, self.ws, st)

    def kernel_launches_per_step(self) -> int:
        """Kernels of this library launched by one forward (route 1, layout 1 to
        3, dispatch 1 unless fused into the gate/up GEMM, each GEMM 1, combine 1,
        shared expert 3)."""
        s = self.shape
        if s.N == 0:
            return 0
        shared = 3 if self.shared is not None else 0  # dense segment + 2 GEMMs
        dispatch = 0 if self.fused_dispatch else 1
        # fused combine: GEMM + finish (the accumulator memset is a copy-engine op)
        down_combine = 2 if self.fuse_combine else 1 + 1
        gate_up = 0 if self.fused_ffn else 1  # the fused FFN is one launch with the down
        return 1 + layout_launches(s) + dispatch + gate_up + down_combine + shared

    def forward_host(self, logits_h, x_h, residual_h, out_h, dev_inputs=None, stream=None):
        """Whole layer from host buffers: copy the step's inputs host->device,
        run moe_layer_forward, copy the output device->host, all on one stream.
        Host tensors should be pinned for the copies to be asynchronous."""
        st = torch.cuda.current_stream() if stream is None else stream
        if dev_inputs is None:
            dev_inputs = (torch.empty_like(logits_h, device="cuda"),
                          torch.empty_like(x_h, device="cuda"),
                          None if residual_h is None else torch.empty_like(residual_h, device="cuda"))
        L_d, x_d, r_d = dev_inputs
        with torch.cuda.stream(st):
            L_d.copy_(logits_h, non_blocking=True)
            x_d.copy_(x_h, non_blocking=True)
            if residual_h is not None:
                r_d.copy_(residual_h, non_blocking=True)
            out = self.forward(L_d, x_d, r_d if residual_h is not None else None, stream=st)
            out_h.copy_(out, non_blocking=True)
        return out_h

    def check_device_errors(self, stream=None):
        st = moe_get_error(self.ws, stream)
        if st != 0:
            raise MoeError(st, "device")


class HostPipeline:
    """Runs one MoELayer over a sequence of host-resident batches with the
    transfers overlapped: while batch i computes on the compute stream, batch
    i+1's inputs are copied host->device on one copy stream and batch i-1's
    output device->host on another.  Two sets of device input/output buffers
    alternate; events order every reuse.  Host tensors should be pinned."""

    def __init__(self, layer: "MoELayer", with_residual=True, device="cuda", graphs=True):
        """graphs: run the layer as one CUDA graph per buffer set, captured here
        (a replay skips the per-kernel launch gaps of calling the layer's
        kernels one by one: 0.08-0.09 ms per step on GB300); a runner without
        capture() (MicrobatchPipeline) is always called directly."""
        s = layer.shape
        self.layer = layer
        self.with_residual = with_residual
        bf = dict(dtype=torch.bfloat16, device=device)
        self.bufs = []
        for _ in range(2):
            # zeros: the capture's warm-up call runs on these before any batch
            self.bufs.append(dict(
                logits=torch.zeros(max(s.N, 1), s.E, dtype=torch.float32, device=device),
                x=torch.zeros(max(s.N, 1), s.H, **bf),
                res=torch.zeros(max(s.N, 1), s.H, **bf) if with_residual else None,
                out=torch.zeros(max(s.N, 1), s.H, **bf)))
        self.h2d = torch.cuda.Stream(device=device)
        self.d2h = torch.cuda.Stream(device=device)
        mk = lambda: [torch.cuda.Event(), torch.cuda.Event()]  # noqa: E731
        self.loaded, self.computed, self.saved = mk(), mk(), mk()
        self.graphs = None
        if graphs and hasattr(layer, "capture") and s.N > 0:
            self.graphs = [layer.capture(b["logits"], b["x"], b["res"], b["out"])
                           for b in self.bufs]

    def run(self, batches, stream=None):
        """batches: iterable of (logits_h, x_h, residual_h or None, out_h).
        Enqueues everything; the caller synchronizes (or waits on `stream`,
        which is made to wait for the last device->host copy)."""
        comp = torch.cuda.current_stream() if stream is None else stream
        self.h2d.wait_stream(comp)
        self.d2h.wait_stream(comp)
        for i, (L_h, x_h, r_h, out_h) in enumerate(batches):
            b = i % 2
            buf = self.bufs[b]
            if i >= 2:
                self.h2d.wait_event(self.computed[b])  # inputs of batch i-2 consumed
            with torch.cuda.stream(self.h2d):
                buf["logits"].copy_(L_h, non_blocking=True)
                buf["x"].copy_(x_h, non_blocking=True)
                if r_h is not None:
                    buf["res"].copy_(r_h, non_blocking=True)
                self.loaded[b].record(self.h2d)
            comp.wait_event(self.loaded[b])
            if i >= 2:
                comp.wait_event(self.saved[b])  # output of batch i-2 copied out
            if self.graphs is not None and (r_h is not None) == self.with_residual:
                with torch.cuda.stream(comp):
                    self.graphs[b].replay()
            else:
                self.layer.forward(buf["logits"], buf["x"],
                                   buf["res"] if r_h is not None else None, out=buf["out"],
                                   stream=comp)
            self.computed[b].record(comp)
            self.d2h.wait_event(self.computed[b])
            with torch.cuda.stream(self.d2h):
                out_h.copy_(buf["out"], non_blocking=True)
                self.saved[b].record(self.d2h)
        comp.wait_stream(self.d2h)


class MicrobatchPipeline:
    """The layer over microbatches of `microbatch` tokens, with the vector-unit
    stages of one microbatch overlapping the tensor-core stages of another
    ("Kernel fusion for expert parallelism", section "Pipelining and three-way
    overlap": while the matrix units multiply microbatch m, the vector units
    route, dispatch and combine its neighbours; buffers are alive per pipeline
    slot, not per microbatch).

    Two streams: `vec` runs route, layout, dispatch and combine; `mat` runs
    the gate/up and down GEMMs (and the shared expert).  Where the layer
    gathers rows inside the gate/up GEMM (dedup expansion, fused plain
    dispatch), the microbatches do the same.  Microbatch
    m uses buffer set m % depth.  Enqueue order on `vec` is A0, A1, C0, A2, C1,
    ... so a set is overwritten only after its previous microbatch's combine
    (which itself waited for that microbatch's GEMMs).  The GEMM CTAs fill the
    SMs' shared memory but leave threads and registers free, so the copy-stage
    blocks run on the same SMs at the same time.  Every token's output is
    computed exactly as by MoELayer.forward (same kernels, same summation
    order), so the results are bit-identical."""

    def __init__(self, shape: Shape, w_gate, w_up, w_down, placement=None, microbatch=2048,
                 depth=2, shared=None, device="cuda", pack=True):
        """pack: as for MoELayer (one packed copy, shared by the buffer sets)."""
        if depth < 2:
            raise ValueError("the two-stream schedule needs at least two buffer sets")
        if pack and shape.weights == "row_major":
            w_gate, w_down = pack_weights(shape, w_gate, w_up, w_down)
            w_up = None
            shape = dataclasses.replace(shape, weights="packed")
        self.shape = shape
        self.mb = max(1, min(microbatch, shape.N))
        self.depth = depth
        self.placement = placement
        self.w = (w_gate, w_up, w_down)
        self.shared = shared
        sub = dataclasses.replace(shape, N=self.mb)
        self.sets = [MoELayer(sub, w_gate, w_up, w_down, placement, device, shared)
                     for _ in range(depth)]
        self.vec = torch.cuda.Stream(device=device)
        self.mat = torch.cuda.Stream(device=device)
        self.gemm_events = None  # optional [(start, end)] per microbatch, on `mat`

    def chunks(self):
        N = self.shape.N
        return [(t0, min(t0 + self.mb, N)) for t0 in range(0, N, self.mb)]

    def forward(self, logits, x, residual=None, out=None, stream=None, gemm_events=None):
        s = self.shape
        comp = torch.cuda.current_stream() if stream is None else stream
        out = out if out is not None else torch.empty(s.N, s.H, dtype=torch.bfloat16,
                                                      device=x.device)
        vec, mat = self.vec, self.mat
        vec.wait_stream(comp)
        mat.wait_stream(comp)
        chunks = self.chunks()
        a_done = [torch.cuda.Event() for _ in chunks]
        b_done = [torch.cuda.Event() for _ in chunks]

        def sub_shape(t0, t1):
            return dataclasses.replace(s, N=t1 - t0)

        def combine(m):
            t0, t1 = chunks[m]
            L = self.sets[m % self.depth]
            sm = sub_shape(t0, t1)
            res = None if residual is None else residual[t0:t1]
            vec.wait_event(b_done[m])
            if self.shared is not None:
                moe_combine_shared(L.y, L.topk_w, L.layout, sm, L.partial, L.y_s, res,
                                   out[t0:t1], vec)
            else:
                moe_combine(L.y, L.topk_w, L.layout, sm, L.partial, res, out[t0:t1], vec)

        for m, (t0, t1) in enumerate(chunks):
            L = self.sets[m % self.depth]
            sm = sub_shape(t0, t1)
            # vector-unit stages of microbatch m
            moe_route(logits[t0:t1], sm, L.topk_ids, L.topk_w, vec)
            moe_dispatch_layout(L.topk_ids, self.placement, sm, L.layout, L.ws, vec)
            # a chunk never has more rows than its buffer set's shape, so a set
            # sized for the unfused form also fits a fused chunk
            fused = moe_layer_skips_dispatch(sm)
            if not fused:
                moe_dispatch(x[t0:t1], L.layout, sm, L.xd, vec)
            a_done[m].record(vec)
            # tensor-core stages of microbatch m
            mat.wait_event(a_done[m])
            if gemm_events is not None:
                gemm_events[m][0].record(mat)
            ffn_fused = moe_layer_fuses_ffn(sm)
            if ffn_fused:
                # the whole expert FFN in one kernel (h on chip)
                src, index = ((L.xd, L.layout["expand_src"]) if s.dedup else
                              (x[t0:t1], L.layout["row_token"]) if fused else (L.xd, None))
                moe_ffn_fused(src, index, L.layout, sm, self.w[0], self.w[1], self.w[2], L.y,
                              L.ws, mat)
            elif s.dedup:
                moe_ffn_gate_up_gather(L.xd, L.layout["expand_src"], L.layout, sm, self.w[0],
                                       self.w[1], L.h, L.ws, mat)
            elif fused:
                moe_ffn_gate_up_gather(x[t0:t1], L.layout["row_token"], L.layout, sm, self.w[0],
                                       self.w[1], L.h, L.ws, mat)
            else:
                moe_ffn_gate_up(L.xd, L.layout, sm, self.w[0], self.w[1], L.h, L.ws, mat)
            if gemm_events is not None:
                gemm_events[m][1].record(mat)
            if not ffn_fused:
                moe_ffn_down(L.h, L.layout, sm, self.w[2], L.y, L.ws, mat)
            if self.shared is not None:
                moe_shared_expert_ffn(x[t0:t1], sm, L.I_shared, *self.shared, L.h_s, L.y_s,
                                      L.ws, mat)
            b_done[m].record(mat)
            # combine of the previous microbatch while this one multiplies
            if m >= 1:
                combine(m - 1)
        combine(len(chunks) - 1)
        comp.wait_stream(vec)
        comp.wait_stream(mat)
        return out

    def check_device_errors(self):
        for L in self.sets:
            L.check_device_errors()

    def kernel_launches_per_step(self) -> int:
        total = 0
        for t0, t1 in self.chunks():
            s = self.shape
            sub = dataclasses.replace(s, N=t1 - t0)
            dispatch = 0 if moe_layer_skips_dispatch(sub) else 1
            ffn = 1 if moe_layer_fuses_ffn(sub) else 2  # one fused launch, or gate/up + down
            total += 1 + layout_launches(sub) + dispatch + ffn + 1 + (
                3 if self.shared is not None else 0)
        return total
