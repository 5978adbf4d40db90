"""Per-stage parity of the CUDA path (through the C ABI) against the oracle:
route, dispatch layout, dispatch and combine.  Integer and copy results are
compared bit for bit; float results within the layer's tolerance."""
import numpy as np
import pytest
import torch

import oracle
from cases import SMALL
from combine_warp_top_gb300 import moe, synth
from gpu_util import assert_close, dev_bf16, dev_i32, host_f64, host_u16

pytestmark = pytest.mark.gpu

CASE_IDS = list(SMALL)


def shape_of(wl, dedup):
    return moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=dedup)


def run_route(L, shape):
    ids = torch.empty(shape.N * shape.k, dtype=torch.int32, device="cuda")
    w = torch.empty(shape.N * shape.k, dtype=torch.float32, device="cuda")
    moe.moe_route(torch.from_numpy(L).cuda(), shape, ids, w)
    torch.cuda.synchronize()
    return ids.view(shape.N, shape.k).cpu().numpy(), w.view(shape.N, shape.k).cpu().numpy()


@pytest.mark.parametrize("name", CASE_IDS)
def test_route_matches_oracle(name):
    wl = SMALL[name]
    L = synth.make_logits(wl)
    ids, w = run_route(L, shape_of(wl, False))
    ref_ids, ref_w = oracle.route(L, wl.k)
    assert np.array_equal(ids, ref_ids)
    np.testing.assert_allclose(w, ref_w, rtol=0, atol=2e-6)


@pytest.mark.parametrize("E,k", [(8, 3), (64, 6), (256, 8), (1024, 32), (7, 7)])
def test_route_ties_break_to_lower_index(E, k):
    # coarse values: many exact ties, including across lanes of the warp
    u = synth.u64(0, 41, 512 * E) % np.uint64(5)
    L = (u.astype(np.float32) * np.float32(0.5)).reshape(512, E)
    L[0, :] = 0.0
    L[1, :] = -0.0
    ids, w = run_route(L, moe.Shape(512, 8, E, k, 1, 8))
    ref_ids, ref_w = oracle.route(L, k)
    assert np.array_equal(ids, ref_ids)
    np.testing.assert_allclose(w, ref_w, rtol=0, atol=2e-6)


def run_layout(ids, placement, shape):
    lay = moe.Layout(shape)
    ws = moe.workspace(shape)
    moe.moe_dispatch_layout(dev_i32(ids), None if placement is None else dev_i32(placement), shape,
                            lay, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    return {n: t.cpu().numpy() for n, t in lay.tensors.items()}


LAYOUT_KEYS = ["expert_counts", "expert_offsets", "rank_offsets", "row_token"]
DEDUP_KEYS = ["dedup_counts", "dedup_offsets", "expand_src"]


def check_layout(got, ref, shape):
    N, k = shape.N, shape.k
    for key in LAYOUT_KEYS:
        assert np.array_equal(got[key][:len(ref[key])], ref[key]), key
    assert np.array_equal(got["pair_row"].reshape(N, k), ref["pair_row"])
    if shape.dedup:
        Rd = ref["n_dedup_rows"]
        assert int(got["n_dedup_rows"][0]) == Rd
        for key in DEDUP_KEYS:
            assert np.array_equal(got[key][:len(ref[key])], ref[key]), key
        assert np.array_equal(got["dedup_row_token"][:Rd], ref["dedup_row_token"])
        assert np.array_equal(got["pair_dedup_row"].reshape(N, k), ref["pair_dedup_row"])


@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("name", CASE_IDS)
def test_layout_bit_exact(name, dedup):
    wl = SMALL[name]
    L = synth.make_logits(wl)
    ids, _ = oracle.route(L, wl.k)
    shape = shape_of(wl, dedup)
    got = run_layout(ids, None, shape)
    check_layout(got, oracle.dispatch_layout(ids, np.arange(wl.E), wl.E, wl.W), shape)


@pytest.mark.parametrize("dedup", [False, True])
def test_layout_permuted_placement(dedup):
    wl = synth.Workload("perm", 700, 64, 32, 4, 64, 8)
    L = synth.make_logits(wl)
    ids, _ = oracle.route(L, wl.k)
    placement = synth.permutation(0, 51, wl.E).astype(np.int32)
    shape = shape_of(wl, dedup)
    got = run_layout(ids, placement, shape)
    check_layout(got, oracle.dispatch_layout(ids, placement, wl.E, wl.W), shape)


# The scatter blocks copy the per-block count tables ([nb][E], then [nb][W])
# into shared memory in 16-byte pieces and sum tall columns in parts: tables
# whose length is not a multiple of four words (the copies' partial tails),
# and tables tall enough (at least 16 blocks) to be split into parts.
@pytest.mark.parametrize("placed", [False, True])
@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("N,E,k,W", [(700, 21, 3, 7), (4400, 7, 3, 7), (5000, 6, 3, 3),
                                     (20000, 12, 4, 4)])
def test_layout_count_table_tails_and_parts(N, E, k, W, dedup, placed):
    wl = synth.Workload("tables", N, 64, E, k, 64, W)
    ids, _ = oracle.route(synth.make_logits(wl), k)
    placement = synth.permutation(0, 52, E).astype(np.int32) if placed else None
    shape = shape_of(wl, dedup)
    got = run_layout(ids, placement, shape)
    ref_placement = placement if placed else np.arange(E)
    check_layout(got, oracle.dispatch_layout(ids, ref_placement, E, W), shape)


@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("name", ["ragged", "wide", "e256", "k32"])
def test_layout_with_a_workspace_off_16_bytes(name, dedup):
    """A workspace that starts 4 bytes past a 16-byte boundary: the count
    tables cannot be copied in 16-byte pieces, so the layout takes its separate
    scan launch; the tables must not change."""
    wl = SMALL[name]
    ids, _ = oracle.route(synth.make_logits(wl), wl.k)
    shape = shape_of(wl, dedup)
    want = run_layout(ids, None, shape)
    n = moe.moe_workspace_bytes(shape)
    big = torch.zeros(n + 16, dtype=torch.uint8, device="cuda")
    ws = big[4:4 + n]
    assert ws.data_ptr() % 16 == 4
    lay = moe.Layout(shape)
    moe.moe_dispatch_layout(dev_i32(ids), None, shape, lay, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    for key, t in lay.tensors.items():
        assert np.array_equal(t.cpu().numpy(), want[key]), key
    check_layout(want, oracle.dispatch_layout(ids, np.arange(wl.E), wl.E, wl.W), shape)


def test_layout_skewed_and_empty_experts():
    # every token on expert 5 and one of {0, 1}: most experts empty, one full
    N, E, k, W = 1000, 16, 2, 4
    ids = np.zeros((N, k), np.int32)
    ids[:, 0] = 5
    ids[:, 1] = np.arange(N) % 2
    ids[7, 1] = 9  # a single-row expert
    shape = moe.Shape(N, 64, E, k, W, 64, dedup=True)
    got = run_layout(ids, None, shape)
    check_layout(got, oracle.dispatch_layout(ids, np.arange(E), E, W), shape)


def test_layout_is_deterministic():
    wl = SMALL["wide"]
    ids, _ = oracle.route(synth.make_logits(wl), wl.k)
    shape = shape_of(wl, True)
    first = run_layout(ids, None, shape)
    for _ in range(5):
        again = run_layout(ids, None, shape)
        for key in first:
            assert np.array_equal(first[key], again[key]), key


@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("name", ["tiny", "ragged", "odd_h", "k_eq_e", "e256"])
def test_dispatch_bit_exact(name, dedup):
    wl = SMALL[name]
    ids, _ = oracle.route(synth.make_logits(wl), wl.k)
    x = synth.make_x(wl)
    shape = shape_of(wl, dedup)
    ref = oracle.dispatch_layout(ids, np.arange(wl.E), wl.E, wl.W)
    lay = moe.Layout(shape)
    ws = moe.workspace(shape)
    moe.moe_dispatch_layout(dev_i32(ids), None, shape, lay, ws)
    rows = shape.R_d_max if dedup else shape.R
    xd = torch.empty(rows, wl.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch(dev_bf16(x), lay, shape, xd)
    torch.cuda.synchronize()
    got = host_u16(xd)
    if dedup:
        Rd = ref["n_dedup_rows"]
        assert np.array_equal(got[:Rd], oracle.dispatch_dedup(x, ref["dedup_row_token"]))
    else:
        assert np.array_equal(got, oracle.dispatch(x, ref["row_token"]))


# long rows whose last step along the row is ragged: H = 2056 (257 16-byte
# chunks) with k = 5 (one chunk per lane per step: 9 steps, the last 1 chunk),
# H = 1032 (129 chunks) with k = 2 (four chunks per lane: 2 steps, the last 1)
LONG_ROWS = {
    "long_k5": synth.Workload("long_k5", 40, 2056, 10, 5, 128, 2),
    "long_k2": synth.Workload("long_k2", 30, 1032, 8, 2, 128, 4),
}


@pytest.mark.parametrize("dedup", [False, True])
@pytest.mark.parametrize("residual", [True, False])
@pytest.mark.parametrize("name", ["tiny", "ragged", "wide", "k_eq_e", "one_rank", "e256",
                                  "long_k5", "long_k2", "k12", "k32"])
def test_combine_matches_oracle(name, dedup, residual):
    wl = {**SMALL, **LONG_ROWS}[name]
    L = synth.make_logits(wl)
    ids, w64 = oracle.route(L, wl.k)
    shape = shape_of(wl, dedup)
    ref = oracle.dispatch_layout(ids, np.arange(wl.E), wl.E, wl.W)
    # expert outputs: any bf16 rows will do for the combine stage
    y = synth.normal_bf16(0, 61, (shape.R, wl.H))
    res = synth.make_residual(wl) if residual else None
    lay = moe.Layout(shape)
    ws = moe.workspace(shape)
    moe.moe_dispatch_layout(dev_i32(ids), None, shape, lay, ws)
    w32 = w64.astype(np.float32)
    partial = torch.empty(shape.R_d_max, wl.H, dtype=torch.bfloat16, device="cuda") if dedup else None
    out = torch.empty(wl.N, wl.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(dev_bf16(y), torch.from_numpy(w32).cuda(), lay, shape, partial,
                    None if res is None else dev_bf16(res), out)
    torch.cuda.synchronize()
    yf = oracle.widen_bf16(y)
    if dedup:
        _, want = oracle.combine_dedup(yf, w32.astype(np.float64), ref["pair_row"],
                                       ref["pair_dedup_row"], ref["n_dedup_rows"], res)
    else:
        want = oracle.combine(yf, w32.astype(np.float64), ref["pair_row"], res)
    assert_close(host_f64(out), want, "combine")


def test_combine_in_place_on_residual():
    wl = SMALL["ragged"]
    ids, w64 = oracle.route(synth.make_logits(wl), wl.k)
    shape = shape_of(wl, False)
    ref = oracle.dispatch_layout(ids, np.arange(wl.E), wl.E, wl.W)
    y = synth.normal_bf16(0, 62, (shape.R, wl.H))
    res = synth.make_residual(wl)
    lay = moe.Layout(shape)
    ws = moe.workspace(shape)
    moe.moe_dispatch_layout(dev_i32(ids), None, shape, lay, ws)
    stream_buf = dev_bf16(res)
    w32 = w64.astype(np.float32)
    moe.moe_combine(dev_bf16(y), torch.from_numpy(w32).cuda(), lay, shape, None, stream_buf,
                    stream_buf)
    torch.cuda.synchronize()
    want = oracle.combine(oracle.widen_bf16(y), w32.astype(np.float64), ref["pair_row"], res)
    assert_close(host_f64(stream_buf), want, "in-place combine")


@pytest.mark.parametrize("residual", [True, False])
@pytest.mark.parametrize("name", ["tiny", "ragged", "wide", "k_eq_e", "one_rank", "e256", "odd_h",
                                  "deep_k", "long_k5", "long_k2", "k12", "k32", "k12_placed",
                                  "k32_placed"])
def test_dedup_combine_one_pass_equals_two_level(name, residual):
    """The one-pass dedup combine (partial = NULL: partials in registers) gives
    the two-level form's output bit for bit, and both match the oracle.  The
    "_placed" cases put the experts on ranks by a seeded permutation, so the
    ranks of a token's experts interleave in its j order."""
    placed = name.endswith("_placed")
    wl = {**SMALL, **LONG_ROWS}[name.removesuffix("_placed")]
    ids, w64 = oracle.route(synth.make_logits(wl), wl.k)
    shape = shape_of(wl, True)
    placement = synth.permutation(0, 53, wl.E).astype(np.int32) if placed else np.arange(wl.E)
    ref = oracle.dispatch_layout(ids, placement, wl.E, wl.W)
    y = synth.normal_bf16(0, 63, (shape.R, wl.H))
    res = synth.make_residual(wl) if residual else None
    lay = moe.Layout(shape)
    ws = moe.workspace(shape)
    moe.moe_dispatch_layout(dev_i32(ids), dev_i32(placement.astype(np.int32)) if placed else None,
                            shape, lay, ws)
    w32 = torch.from_numpy(w64.astype(np.float32)).cuda()
    partial = torch.empty(shape.R_d_max, wl.H, dtype=torch.bfloat16, device="cuda")
    out2 = torch.empty(wl.N, wl.H, dtype=torch.bfloat16, device="cuda")
    out1 = torch.empty_like(out2)
    r = None if res is None else dev_bf16(res)
    moe.moe_combine(dev_bf16(y), w32, lay, shape, partial, r, out2)
    moe.moe_combine(dev_bf16(y), w32, lay, shape, None, r, out1)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    _, want = oracle.combine_dedup(oracle.widen_bf16(y), w64.astype(np.float32).astype(np.float64),
                                   ref["pair_row"], ref["pair_dedup_row"], ref["n_dedup_rows"], res)
    assert_close(host_f64(out1), want, "one-pass dedup combine")
