"""Pins of the oracle's expert FFN and combine.

Sources: FarSkip-Collective Sec. 2.1 (MoE(A) = sum_j G(A)_j MLP^j(A), gated
MLP) and "Kernel fusion for expert parallelism", sections "AllGather-
ReduceScatter" (every rank evaluates its experts on every token, zero where a
token is not routed, and the owner sums) and "Fusing the layer into one
kernel" (stages 4-7: gate/up MatMul, SwiGLU, down MatMul, weighted reduce).
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from combine_warp_top_gb300 import synth


def make_case(N=24, H=32, E=6, k=3, I=40, W=3, seed=0, placement=None):
    wl = synth.Workload("t", N, H, E, k, I, W)
    L = synth.make_logits(wl, seed)
    x = synth.make_x(wl, seed)
    wg = synth.make_weight(wl, "gate", seed)
    wu = synth.make_weight(wl, "up", seed)
    wd = synth.make_weight(wl, "down", seed)
    res = synth.make_residual(wl, seed)
    return L, x, wg, wu, wd, res, wl


def check_dense_brute_force(layer_fn):
    for dedup in (False, True):
        for k, W in ((1, 2), (2, 3), (3, 6), (6, 1)):
            L, x, wg, wu, wd, res, wl = make_case(k=k, W=W, seed=k + 10 * W)
            sparse = layer_fn(L, x, wg, wu, wd, k, W, residual=res, dedup=dedup)["out"]
            dense = oracle.dense_forward(L, x, wg, wu, wd, k, residual=res)
            np.testing.assert_allclose(sparse, dense, rtol=1e-12, atol=1e-12)


def check_single_expert_is_plain_swiglu(layer_fn):
    """k = E = 1, w = 1: the layer is residual + SwiGLU MLP, written here with
    torch's nn.Linear convention y = x A^T and F.silu (float64)."""
    L, x, wg, wu, wd, res, wl = make_case(N=17, H=24, E=1, k=1, I=40, W=1, seed=3)
    got = layer_fn(L, x, wg, wu, wd, 1, 1, residual=res)["out"]
    X = torch.from_numpy(oracle.widen_bf16(x))
    g = F.linear(X, torch.from_numpy(oracle.widen_bf16(wg[0])))
    u = F.linear(X, torch.from_numpy(oracle.widen_bf16(wu[0])))
    y = F.linear(F.silu(g) * u, torch.from_numpy(oracle.widen_bf16(wd[0])))
    want = (torch.from_numpy(oracle.widen_bf16(res)) + y).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def check_two_experts_by_hand(layer_fn):
    """E = 2, k = 2 on one token: out = res + w0 MLP^{e0}(x) + w1 MLP^{e1}(x),
    with both MLPs and the weights computed by hand in torch."""
    L = np.array([[0.3, 1.1]], np.float32)
    _, x, wg, wu, wd, res, wl = make_case(N=1, H=16, E=2, k=2, I=8, W=2, seed=4)
    got = layer_fn(L, x, wg, wu, wd, 2, 2, residual=res)["out"]
    X = torch.from_numpy(oracle.widen_bf16(x))

    def mlp(e):
        g = F.linear(X, torch.from_numpy(oracle.widen_bf16(wg[e])))
        u = F.linear(X, torch.from_numpy(oracle.widen_bf16(wu[e])))
        return F.linear(F.silu(g) * u, torch.from_numpy(oracle.widen_bf16(wd[e])))

    w1 = 1.0 / (1.0 + np.exp(0.3 - 1.1))  # expert 1 has the larger logit
    want = torch.from_numpy(oracle.widen_bf16(res)) + w1 * mlp(1) + (1 - w1) * mlp(0)
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-12, atol=1e-12)


def check_zero_down_projection_leaves_residual(layer_fn):
    L, x, wg, wu, wd, res, wl = make_case(seed=5)
    out = layer_fn(L, x, wg, wu, np.zeros_like(wd), wl.k, wl.W, residual=res)["out"]
    assert np.array_equal(out, oracle.widen_bf16(res))
    out = layer_fn(L, x, np.zeros_like(wg), wu, wd, wl.k, wl.W, residual=None)["out"]
    assert np.array_equal(out, np.zeros_like(out))  # SiLU(0) = 0


PINS = [check_dense_brute_force, check_single_expert_is_plain_swiglu, check_two_experts_by_hand,
        check_zero_down_projection_leaves_residual]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_ffn_pins(pin):
    pin(oracle.layer_forward)


def test_dedup_combine_equals_plain_combine():
    """The two-level (per-rank partial, then owner) sum equals the plain sum up
    to float reassociation, and every partial row belongs to one (token, rank)."""
    L, x, wg, wu, wd, res, wl = make_case(N=40, E=8, k=4, W=4, seed=6)
    a = oracle.layer_forward(L, x, wg, wu, wd, 4, 4, residual=res, dedup=False)
    b = oracle.layer_forward(L, x, wg, wu, wd, 4, 4, residual=res, dedup=True)
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-13, atol=1e-13)
    assert b["partial"].shape[0] == b["layout"]["n_dedup_rows"]
    # dedup dispatch + expansion rebuilds exactly the plain expert-major rows
    assert np.array_equal(a["xd"], b["xd"])


def test_token_outputs_match_layer():
    L, x, wg, wu, wd, res, wl = make_case(N=30, E=6, k=2, W=2, seed=7)
    full = oracle.layer_forward(L, x, wg, wu, wd, 2, 2, residual=res)
    ids, w = full["topk_ids"], full["topk_w"]
    sample = np.array([0, 7, 29])
    out, y_rows = oracle.token_outputs(x[sample], ids[sample], w[sample],
                                       lambda e: (wg[e], wu[e], wd[e]), res[sample])
    np.testing.assert_allclose(out, full["out"][sample], rtol=1e-12, atol=1e-12)
    for si, t in enumerate(sample):
        for j in range(2):
            np.testing.assert_allclose(y_rows[si, j], full["y"][full["layout"]["pair_row"][t, j]],
                                       rtol=1e-12, atol=1e-12)


def test_expert_with_no_rows_and_ragged_segments():
    # E=8, k=1 on 5 tokens leaves most experts empty
    L, x, wg, wu, wd, res, wl = make_case(N=5, E=8, k=1, W=4, seed=8)
    r = oracle.layer_forward(L, x, wg, wu, wd, 1, 4, residual=res)
    dense = oracle.dense_forward(L, x, wg, wu, wd, 1, residual=res)
    np.testing.assert_allclose(r["out"], dense, rtol=1e-12, atol=1e-12)
    assert (r["layout"]["expert_counts"] == 0).any()


def check_shared_expert_is_added_to_every_token(layer_fn):
    """With the routed down projections zeroed, the layer is residual + the
    shared SwiGLU MLP, written here with torch's F.linear / F.silu."""
    L, x, wg, wu, wd, res, wl = make_case(N=20, H=24, E=4, k=2, I=16, W=2, seed=9)
    ws_ = synth.Workload("s", 20, 24, 1, 1, 40, 1)
    shared = tuple(synth.make_weight(ws_, m, seed=9)[0] for m in ("gate", "up", "down"))
    got = layer_fn(L, x, wg, wu, np.zeros_like(wd), 2, 2, residual=res, shared=shared)["out"]
    X = torch.from_numpy(oracle.widen_bf16(x))
    g = F.linear(X, torch.from_numpy(oracle.widen_bf16(shared[0])))
    u = F.linear(X, torch.from_numpy(oracle.widen_bf16(shared[1])))
    y = F.linear(F.silu(g) * u, torch.from_numpy(oracle.widen_bf16(shared[2])))
    want = torch.from_numpy(oracle.widen_bf16(res)) + y
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-12, atol=1e-12)
    # and with routed experts: shared part and routed part add
    both = layer_fn(L, x, wg, wu, wd, 2, 2, residual=res, shared=shared)["out"]
    routed = layer_fn(L, x, wg, wu, wd, 2, 2, residual=res)["out"]
    np.testing.assert_allclose(both - routed, y.numpy(), rtol=1e-10, atol=1e-12)


def test_shared_expert_pin():
    check_shared_expert_is_added_to_every_token(oracle.layer_forward)
