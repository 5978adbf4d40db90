"""Shared helpers of the GPU parity tests: host<->device marshalling of the
seeded inputs and the tolerance of the layer's floating-point outputs."""
import numpy as np
import torch

# Tolerance of the layer's float outputs against the float64 oracle:
# max |got - ref| <= 2e-2 * max |ref| and sum |got - ref| / sum |ref| <= 5e-3.
MAX_ABS_FRAC = 2e-2
MEAN_REL = 5e-3


def dev_bf16(a_u16):
    return torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).view(torch.bfloat16).cuda()


def host_u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def assert_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    scale = np.abs(ref).max()
    assert err.max() <= MAX_ABS_FRAC * scale + 1e-30, f"{what}: max|err| {err.max():.4g} vs max|ref| {scale:.4g}"
    denom = np.abs(ref).sum()
    if denom > 0:
        rel = err.sum() / denom
        assert rel <= MEAN_REL, f"{what}: mean relative error {rel:.4g}"
