"""Parity of the whole layer on seeded random shapes: sizes, expert counts,
rank counts, top-k, routing skew, dedup, placement, GEMM kernel (the fused
expert FFN included where H <= 256) and combine form
are drawn together, so that combinations no hand-picked case names are checked
against the oracle too (ids, counts and R_d exactly, out within the layer's
float tolerance).

Shape rules drawn from: 1 <= N <= 700; H and I multiples of 8 up to 512 and
320; E in 1..64 or 128 / 256; W a divisor of E; 1 <= k <= min(E, 12);
E * H * I <= 2^22 so that the oracle's float64 weights stay small."""
import numpy as np
import pytest
import torch

import oracle
from combine_warp_top_gb300 import moe, synth
from gpu_util import assert_close, dev_bf16, dev_i32, host_f64

pytestmark = pytest.mark.gpu

CASES = 64


def draw_case(i):
    rng = np.random.default_rng(1000 + i)
    while True:
        E = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64, 128, 256]))
        H = 8 * int(rng.integers(1, 65))
        I = 8 * int(rng.integers(1, 41))
        if E * H * I <= (1 << 22):
            break
    divisors = [w for w in range(1, E + 1) if E % w == 0]
    W = int(rng.choice(divisors))
    k = int(rng.integers(1, min(E, 12) + 1))
    N = int(rng.integers(1, 701))
    logits = "zipf" if rng.random() < 0.5 else "iid"
    wl = synth.Workload(f"rand{i}", N, H, E, k, I, W, logits=logits,
                        zipf_alpha=1.2 if logits == "zipf" else 0.0)
    dedup = bool(rng.random() < 0.5)
    placed = bool(rng.random() < 0.5) and E > 1
    gemm = str(rng.choice(["auto", "single", "pair", "fused"]))
    if gemm == "fused" and H > 256:  # the fused FFN keeps a 128 x H tile of y in TMEM
        gemm = "auto"
    fuse = (not dedup) and gemm != "fused" and bool(rng.random() < 0.25)
    residual = bool(rng.random() < 0.8)
    return wl, dedup, placed, gemm, fuse, residual


@pytest.mark.parametrize("i", range(CASES))
def test_layer_random_shape(i):
    wl, dedup, placed, gemm, fuse, residual = draw_case(i)
    N = wl.N
    placement = synth.permutation(i, 53, wl.E).astype(np.int32) if placed else None
    wg, wu, wd = (synth.make_weight(wl, w) for w in ("gate", "up", "down"))
    shape = moe.Shape(N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup, gemm=gemm)
    layer = moe.MoELayer(shape, dev_bf16(wg), dev_bf16(wu), dev_bf16(wd),
                         None if placement is None else dev_i32(placement), fuse_combine=fuse)
    L = synth.make_logits(wl, seed=i)
    x = synth.make_x(wl, seed=i)
    res = synth.make_residual(wl, seed=i) if residual else None
    out = layer.forward(torch.from_numpy(L).cuda(), dev_bf16(x),
                        None if res is None else dev_bf16(res))
    torch.cuda.synchronize()
    layer.check_device_errors()
    ref = oracle.layer_forward(L, x, wg, wu, wd, wl.k, wl.W, placement=placement, residual=res,
                               dedup=dedup)
    what = (f"N={N} H={wl.H} E={wl.E} k={wl.k} W={wl.W} I={wl.I} {wl.logits} dedup={dedup} "
            f"placed={placed} gemm={gemm} fuse={fuse} residual={residual}")
    assert np.array_equal(layer.topk_ids.view(N, wl.k).cpu().numpy(), ref["topk_ids"]), what
    assert np.array_equal(layer.layout["expert_counts"].cpu().numpy(),
                          ref["layout"]["expert_counts"]), what
    if dedup:
        assert int(layer.layout["n_dedup_rows"].item()) == ref["layout"]["n_dedup_rows"], what
    assert_close(host_f64(out), ref["out"], what)
