"""Seeded synthetic workloads for the MoE layer.

This module generates every input of the layer (router logits, token rows,
expert weights, residual stream, placement permutation) from counter-based
SplitMix64 streams (definition in ``synth.c``). It holds none of the method's
arithmetic: the oracle and the CUDA path both receive its arrays unchanged.

Sub-streams of one seed:
  1 router logits (normal part)   2 token rows x      3 gate weights Wg
  4 up weights Wu                 5 down weights Wd   6 residual stream
  7 expert permutation (hot pairs / Zipf ranks)       8 hot-token shuffle
  9 hot-pair choice per hot token

The five workloads follow the shapes and value distributions that the three
pages' MoE models motivate (DeepSeek-V3, Mixtral, the correlated-routing
model of "Expert Coupling", a Zipf-skewed load); no dataset, trace or trained
weight is used anywhere.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

STREAM_LOGITS, STREAM_X, STREAM_WG, STREAM_WU, STREAM_WD, STREAM_RES = 1, 2, 3, 4, 5, 6
STREAM_EXPERT_PERM, STREAM_HOT_TOKENS, STREAM_HOT_PAIR = 7, 8, 9


def build_lib(force: bool = False) -> str:
    """Compile synth.c into an in-tree shared library (host code, any arch)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_GPU_SRC = os.path.join(_HERE, "synth_gpu.cu")
_GPU_LIB = os.path.join(_HERE, "libsynth_gpu.so")
_gpu_lib = None


def build_gpu_lib(force: bool = False) -> str:
    """Compile the device-side twin of the normal_bf16 stream (sm_103a)."""
    if force or not os.path.exists(_GPU_LIB) or os.path.getmtime(_GPU_LIB) < os.path.getmtime(_GPU_SRC):
        tmp = _GPU_LIB + f".tmp{os.getpid()}"
        nvcc = "nvcc" if subprocess.run(["which", "nvcc"], capture_output=True).returncode == 0 \
            else "/usr/local/cuda/bin/nvcc"
        subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                               "-shared", "-Xcompiler", "-fPIC", "-o", tmp, _GPU_SRC,
                               "-cudart", "static"])
        os.replace(tmp, _GPU_LIB)
    return _GPU_LIB


def _get_gpu():
    global _gpu_lib
    with _lock:
        if _gpu_lib is None:
            lib = ctypes.CDLL(build_gpu_lib())
            lib.synth_normal_bf16_device.argtypes = [ctypes.c_uint64, ctypes.c_uint64,
                                                     ctypes.c_uint64, ctypes.c_int64,
                                                     ctypes.c_double, ctypes.c_double,
                                                     ctypes.c_void_p, ctypes.c_void_p]
            lib.synth_normal_bf16_device.restype = ctypes.c_int
            _gpu_lib = lib
    return _gpu_lib


def normal_bf16_device(out, seed, stream, mean=0.0, std=1.0, offset=0):
    """Fill a torch bf16 CUDA tensor with the normal_bf16 stream (device twin)."""
    import torch
    assert out.is_cuda and out.dtype == torch.bfloat16 and out.is_contiguous()
    rc = _get_gpu().synth_normal_bf16_device(seed, stream, offset, out.numel(), mean, std,
                                             out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    if rc != 0:
        raise RuntimeError(f"device generator launch failed ({rc})")
    return out


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_lib())
            u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.synth_u64.argtypes = [u64, u64, u64, i64, vp]
            lib.synth_uniform_f64.argtypes = [u64, u64, u64, i64, vp]
            for f in (lib.synth_normal_f64, lib.synth_normal_f32, lib.synth_normal_bf16):
                f.argtypes = [u64, u64, u64, i64, dbl, dbl, vp]
            lib.synth_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def threads() -> int:
    return int(_get().synth_threads())


# --- raw fills (write into caller memory: numpy array or raw host pointer) -------------

def _ptr(out):
    if isinstance(out, np.ndarray):
        assert out.flags["C_CONTIGUOUS"]
        return out.ctypes.data, out.size
    raise TypeError("expected a C-contiguous numpy array")


def u64(seed, stream, n, offset=0):
    out = np.empty(n, np.uint64)
    _get().synth_u64(seed, stream, offset, n, out.ctypes.data)
    return out


def uniform(seed, stream, n, offset=0):
    out = np.empty(n, np.float64)
    _get().synth_uniform_f64(seed, stream, offset, n, out.ctypes.data)
    return out


def normal_f64(seed, stream, n, mean=0.0, std=1.0, offset=0):
    out = np.empty(n, np.float64)
    _get().synth_normal_f64(seed, stream, offset, n, mean, std, out.ctypes.data)
    return out


def normal_f32(seed, stream, shape, mean=0.0, std=1.0, offset=0, out=None):
    out = np.empty(shape, np.float32) if out is None else out
    p, n = _ptr(out)
    _get().synth_normal_f32(seed, stream, offset, n, mean, std, p)
    return out


def normal_bf16(seed, stream, shape, mean=0.0, std=1.0, offset=0, out=None):
    """bf16 values returned as their uint16 bit patterns."""
    out = np.empty(shape, np.uint16) if out is None else out
    p, n = _ptr(out)
    _get().synth_normal_bf16(seed, stream, offset, n, mean, std, p)
    return out


def normal_bf16_ptr(ptr: int, n: int, seed, stream, mean=0.0, std=1.0, offset=0):
    """Fill n bf16 values at a raw host address (e.g. a pinned torch tensor)."""
    _get().synth_normal_bf16(seed, stream, offset, n, mean, std, ptr)


def permutation(seed, stream, n, offset=0):
    """Fisher-Yates shuffle of range(n); draw i picks j = x_i mod (n - i) + i."""
    draws = u64(seed, stream, max(n - 1, 0), offset)
    perm = np.arange(n, dtype=np.int64)
    for i in range(n - 1):
        j = i + int(draws[i] % np.uint64(n - i))
        perm[i], perm[j] = perm[j], perm[i]
    return perm


# --- workloads -------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    N: int
    H: int
    E: int
    k: int
    I: int
    W: int
    logits: str = "iid"            # iid | hot_pairs | zipf
    placement: str = "contiguous"  # contiguous | correlated
    dedup: bool = False
    residual: bool = True
    hot_pairs: int = 0
    hot_frac: float = 0.0
    hot_boost: float = 0.0
    zipf_alpha: float = 0.0
    describe: str = ""

    def shape_dict(self):
        return dict(N=self.N, H=self.H, E=self.E, k=self.k, W=self.W, I=self.I, dedup=int(self.dedup))


WORKLOADS = {
    "tiny": Workload("tiny", 64, 128, 8, 2, 256, 2,
                     describe="tiny MoE layer N=64 H=128 E=8 top-2 I=256 W=2"),
    "deepseek_v3": Workload("deepseek_v3", 4096, 7168, 256, 8, 2048, 8,
                            describe="DeepSeek-V3-shaped layer N=4096 H=7168 E=256 top-8 I=2048 W=8"),
    "mixtral": Workload("mixtral", 8192, 4096, 8, 2, 14336, 8,
                        describe="Mixtral-shaped layer N=8192 H=4096 E=8 top-2 I=14336 W=8"),
    "correlated_contiguous": Workload(
        "correlated_contiguous", 16384, 2048, 64, 6, 1408, 32, logits="hot_pairs",
        placement="contiguous", dedup=True, hot_pairs=20, hot_frac=0.42, hot_boost=4.0,
        describe="correlated-routing layer N=16384 H=2048 E=64 top-6 I=1408 W=32, contiguous placement, dedup"),
    "correlated_placed": Workload(
        "correlated_placed", 16384, 2048, 64, 6, 1408, 32, logits="hot_pairs",
        placement="correlated", dedup=True, hot_pairs=20, hot_frac=0.42, hot_boost=4.0,
        describe="correlated-routing layer N=16384 H=2048 E=64 top-6 I=1408 W=32, hot pairs co-located, dedup"),
    "skewed": Workload("skewed", 32768, 4096, 128, 8, 1536, 16, logits="zipf", zipf_alpha=1.2,
                       describe="Zipf(1.2)-skewed layer N=32768 H=4096 E=128 top-8 I=1536 W=16"),
}


def hot_pairs(wl: Workload, seed=0):
    """The planted expert pairs: the first 2*P entries of a seeded expert permutation."""
    perm = permutation(seed, STREAM_EXPERT_PERM, wl.E)
    return perm[: 2 * wl.hot_pairs].reshape(wl.hot_pairs, 2)


def make_logits(wl: Workload, seed=0, N=None):
    """Router logits fp32 [N, E].

    iid:       N(0, 1).
    hot_pairs: N(0, 1); round(hot_frac * N) tokens (a seeded shuffle) each get one
               of the planted pairs (seeded uniform choice), both logits + hot_boost.
    zipf:      N(0, 1) + ln p_e, p_e proportional to r^-alpha where r is the
               1-based rank of expert e in a seeded permutation.
    """
    N = wl.N if N is None else N
    if wl.logits == "iid":
        return normal_f32(seed, STREAM_LOGITS, (N, wl.E))
    if wl.logits == "hot_pairs":
        L = normal_f32(seed, STREAM_LOGITS, (N, wl.E))
        pairs = hot_pairs(wl, seed)
        n_hot = int(round(wl.hot_frac * N))
        hot_tokens = permutation(seed, STREAM_HOT_TOKENS, N)[:n_hot]
        choice = u64(seed, STREAM_HOT_PAIR, n_hot) % np.uint64(wl.hot_pairs)
        boost = np.float32(wl.hot_boost)
        for t, c in zip(hot_tokens, choice):
            a, b = pairs[int(c)]
            L[t, a] = L[t, a] + boost
            L[t, b] = L[t, b] + boost
        return L
    if wl.logits == "zipf":
        perm = permutation(seed, STREAM_EXPERT_PERM, wl.E)
        rank = np.empty(wl.E, np.float64)
        rank[perm] = np.arange(1, wl.E + 1, dtype=np.float64)
        p = rank ** (-wl.zipf_alpha)
        p = p / p.sum()
        n = normal_f64(seed, STREAM_LOGITS, N * wl.E).reshape(N, wl.E)
        return (n + np.log(p)[None, :]).astype(np.float32)
    raise ValueError(wl.logits)


def make_placement(wl: Workload, seed=0):
    """Placement permutation pi [E] int32: pi[p] = global expert held at slot p;
    slot p belongs to rank p // (E / W).

    contiguous: identity. correlated: rank i < P holds planted pair i, and the
    remaining experts fill the later slots in ascending order.
    """
    if wl.placement == "contiguous":
        return np.arange(wl.E, dtype=np.int32)
    pairs = hot_pairs(wl, seed)
    first = [int(e) for pr in pairs for e in pr]
    rest = sorted(set(range(wl.E)) - set(first))
    return np.array(first + rest, dtype=np.int32)


def make_x(wl: Workload, seed=0, N=None):
    N = wl.N if N is None else N
    return normal_bf16(seed, STREAM_X, (N, wl.H))


def make_residual(wl: Workload, seed=0, N=None):
    N = wl.N if N is None else N
    return normal_bf16(seed, STREAM_RES, (N, wl.H))


def make_weight(wl: Workload, which: str, seed=0, experts=None):
    """Expert weights as bf16 bit patterns, nn.Linear layout [out, in]:
    gate/up [E, I, H], down [E, H, I]; ~N(0, 0.02).  ``experts`` selects a
    subset (generated from the same counters as the full tensor)."""
    stream = {"gate": STREAM_WG, "up": STREAM_WU, "down": STREAM_WD}[which]
    rows, cols = (wl.I, wl.H) if which in ("gate", "up") else (wl.H, wl.I)
    per = rows * cols
    if experts is None:
        return normal_bf16(seed, stream, (wl.E, rows, cols), std=0.02)
    out = np.empty((len(experts), rows, cols), np.uint16)
    for i, e in enumerate(experts):
        normal_bf16(seed, stream, (rows, cols), std=0.02, offset=int(e) * per, out=out[i])
    return out


def make_weight_device(wl: Workload, which: str, seed=0):
    """Same tensor as make_weight, generated directly in device memory."""
    import torch
    stream = {"gate": STREAM_WG, "up": STREAM_WU, "down": STREAM_WD}[which]
    rows, cols = (wl.I, wl.H) if which in ("gate", "up") else (wl.H, wl.I)
    out = torch.empty(wl.E, rows, cols, dtype=torch.bfloat16, device="cuda")
    return normal_bf16_device(out, seed, stream, std=0.02)


def bf16_to_f64(a):
    """Exact widening of bf16 bit patterns to float64."""
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_to_f32(a):
    return (a.astype(np.uint32) << 16).view(np.float32)
