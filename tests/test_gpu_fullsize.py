"""Parity at the full sizes of the five benchmark workloads, in the launch
configuration bench.py times (one moe_layer_forward per step, weights filled
in device memory).

Integer results are checked in full against the oracle: routing ids, every
layout table, the dedup row count.  Copies are checked bit for bit on sampled
rows.  Float outputs are checked on sampled tokens, each recomputed by the
oracle straight from the MoE definition with host-generated weights of the
experts those tokens use (each expert's weights generated and widened once).

Tile-coverage rule of the float check: the sampled tokens are chosen so that
every (expert, 128-row block) tile of the plain expert-major rows holds at
least one checked row, and the last row of every expert's segment (its ragged
tail) is checked.  A 128-row block is the single-CTA kernel's tile and half of
the CTA-pair kernel's 256-row tile (both start at the segment's first row), so
every tile of either GEMM kernel, in every n-block (a checked row is checked
in all its columns), reaches the check, and so does every token block of the
combine through the checked tokens' rows."""
import numpy as np
import pytest
import torch

import oracle
from combine_warp_top_gb300 import moe, synth
from gpu_util import assert_close, dev_i32, host_f64, host_u16

pytestmark = pytest.mark.gpu

WORKLOADS = ["deepseek_v3", "mixtral", "correlated_contiguous", "correlated_placed", "skewed"]
# tokens sampled for the option checks that are not the benchmarked path
SAMPLES = {"deepseek_v3": 8, "correlated_placed": 24}
BLOCK = 128


def tile_covering_tokens(ref, N, k, rng, block=BLOCK):
    """Tokens whose rows reach every (expert, block-row) tile of the plain
    expert-major rows and every expert's last row: first the token of each
    non-empty expert's last row, then, visiting the tiles in a seeded random
    order, the token of a random row of each tile not yet reached (a token
    reaches the tiles of all k of its rows).  Returns (tokens, tile count)."""
    off, cnt = ref["expert_offsets"], ref["expert_counts"]
    row_token, pair_row = ref["row_token"], ref["pair_row"]
    tile_of_row = np.empty(N * k, np.int64)
    tiles = []  # (first row, last row) of every tile
    for e in range(len(cnt)):
        a, n = int(off[e]), int(cnt[e])
        for b0 in range(0, n, block):
            tile_of_row[a + b0:a + min(n, b0 + block)] = len(tiles)
            tiles.append((a + b0, a + min(n, b0 + block) - 1))
    covered = np.zeros(len(tiles), bool)
    chosen = [0, N - 1] + [int(row_token[int(off[e]) + int(cnt[e]) - 1])
                           for e in range(len(cnt)) if cnt[e] > 0]
    for t in chosen:
        covered[tile_of_row[pair_row[t]]] = True
    for i in rng.permutation(len(tiles)):
        if not covered[i]:
            first, last = tiles[i]
            t = int(row_token[int(rng.integers(first, last + 1))])
            chosen.append(t)
            covered[tile_of_row[pair_row[t]]] = True
    assert covered.all()
    return np.unique(np.array(chosen, np.int64)), len(tiles)


def prefetched_weights(wl, experts, asked, ahead=2):
    """weights_of(e) for oracle.token_outputs, which asks for the experts in
    ascending order: host-generated bf16 weights of expert e, the next experts'
    generated on a worker thread while the oracle works on this one."""
    from concurrent.futures import ThreadPoolExecutor
    order = [int(e) for e in sorted(experts)]
    pool = ThreadPoolExecutor(1)
    futures = {}

    def gen(e):
        return tuple(synth.make_weight(wl, m, experts=[e])[0] for m in ("gate", "up", "down"))

    def submit(i):
        if i < len(order) and order[i] not in futures:
            futures[order[i]] = pool.submit(gen, order[i])

    for i in range(ahead):
        submit(i)

    def weights_of(e):
        asked.append(e)
        i = order.index(e)
        for j in range(i, i + ahead + 1):
            submit(j)
        return futures.pop(e).result()

    return weights_of


def bf16_host(a):
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)


@pytest.fixture(scope="module")
def runs():
    return {}


def run_full(name, fuse_combine=False):
    wl = synth.WORKLOADS[name]
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=wl.dedup)
    placement = synth.make_placement(wl)
    pl_d = None if wl.placement == "contiguous" else dev_i32(placement)
    layer = moe.MoELayer(shape, synth.make_weight_device(wl, "gate"),
                         synth.make_weight_device(wl, "up"), synth.make_weight_device(wl, "down"),
                         pl_d, fuse_combine=fuse_combine)
    L = synth.make_logits(wl)
    x = synth.make_x(wl)
    res = synth.make_residual(wl)
    out = layer.forward(torch.from_numpy(L).cuda(), bf16_host(x).cuda(), bf16_host(res).cuda())
    torch.cuda.synchronize()
    layer.check_device_errors()
    return wl, layer, L, x, res, placement, out


@pytest.mark.parametrize("name", WORKLOADS)
def test_full_size_workload(name):
    wl, layer, L, x, res, placement, out = run_full(name)
    N, k = wl.N, wl.k
    # routing: ids bit-exact, weights to fp32 rounding
    ids = layer.topk_ids.view(N, k).cpu().numpy()
    w = layer.topk_w.view(N, k).cpu().numpy()
    ref_ids, ref_w = oracle.route(L, k)
    assert np.array_equal(ids, ref_ids)
    np.testing.assert_allclose(w, ref_w, rtol=0, atol=2e-6)
    # every layout table, bit-exact
    ref = oracle.dispatch_layout(ref_ids, placement, wl.E, wl.W)
    got = {n: t.cpu().numpy() for n, t in layer.layout.tensors.items()}
    for key in ("expert_counts", "expert_offsets", "rank_offsets", "row_token"):
        assert np.array_equal(got[key][:len(ref[key])], ref[key]), key
    assert np.array_equal(got["pair_row"].reshape(N, k), ref["pair_row"])
    rng = np.random.default_rng(7)
    if wl.dedup:
        Rd = ref["n_dedup_rows"]
        assert int(got["n_dedup_rows"][0]) == Rd
        for key in ("dedup_counts", "dedup_offsets", "expand_src"):
            assert np.array_equal(got[key][:len(ref[key])], ref[key]), key
        assert np.array_equal(got["dedup_row_token"][:Rd], ref["dedup_row_token"])
        assert np.array_equal(got["pair_dedup_row"].reshape(N, k), ref["pair_dedup_row"])
        rows = rng.choice(Rd, size=min(512, Rd), replace=False)
        xd = layer.xd[torch.from_numpy(rows).cuda()]
        assert np.array_equal(host_u16(xd), x[ref["dedup_row_token"][rows]])
    else:
        xd_buf = layer.xd
        if layer.fused_dispatch:
            # the layer gathered its rows inside the GEMM; the dispatch kernel
            # itself is checked at this size on its own buffer
            xd_buf = torch.empty(N * k, wl.H, dtype=torch.bfloat16, device="cuda")
            moe.moe_dispatch(bf16_host(x).cuda(), layer.layout, layer.shape, xd_buf)
            torch.cuda.synchronize()
        rows = rng.choice(N * k, size=512, replace=False)
        xd = xd_buf[torch.from_numpy(rows).cuda()]
        assert np.array_equal(host_u16(xd), x[ref["row_token"][rows]])
    # every output finite (a property at any size)
    assert bool(torch.isfinite(out.float()).all())
    # float outputs on the tokens that reach every GEMM tile (module docstring)
    toks, n_tiles = tile_covering_tokens(ref, N, k, rng)
    # each expert's weights are generated and widened once: token_outputs asks
    # for every expert once, in ascending order
    asked = []
    weights_of = prefetched_weights(wl, np.unique(ref_ids[toks]), asked)
    want, y_want = oracle.token_outputs(x[toks], ref_ids[toks], ref_w[toks], weights_of, res[toks])
    assert len(asked) == len(set(asked))
    print(f"{name}: {len(toks)} tokens checked, {n_tiles} tiles, {len(asked)} experts")
    got_out = host_f64(out[torch.from_numpy(toks).cuda()])
    assert_close(got_out, want, f"{name} out")
    # the MoE delta alone: rerun without the residual (subtracting it from the
    # bf16 total would measure the total's rounding against a smaller delta)
    delta = layer.forward(torch.from_numpy(L).cuda(), bf16_host(x).cuda(), None)
    torch.cuda.synchronize()
    got_delta = host_f64(delta[torch.from_numpy(toks).cuda()])
    assert_close(got_delta, want - oracle.widen_bf16(res[toks]), f"{name} MoE delta")
    pr = ref["pair_row"][toks].reshape(-1)
    y_got = host_f64(layer.y[torch.from_numpy(pr.astype(np.int64)).cuda()])
    assert_close(y_got, y_want.reshape(-1, wl.H), f"{name} y rows")


@pytest.mark.parametrize("name", ["deepseek_v3", "correlated_placed"])
def test_full_size_fused_combine(name):
    """The combine fused into the down GEMM's epilogue at full size, on
    sampled tokens recomputed by the oracle."""
    wl, layer, L, x, res, placement, out = run_full(name, fuse_combine=True)
    N, k = wl.N, wl.k
    ids = layer.topk_ids.view(N, k).cpu().numpy()
    w = layer.topk_w.view(N, k).cpu().numpy()
    ref_ids, ref_w = oracle.route(L, k)
    assert np.array_equal(ids, ref_ids)
    rng = np.random.default_rng(11)
    n = SAMPLES[wl.name]
    toks = np.unique(np.concatenate([[0, N - 1], rng.choice(N, size=n - 2, replace=False)]))

    def weights_of(e):
        return tuple(synth.make_weight(wl, m, experts=[e])[0] for m in ("gate", "up", "down"))

    want, _ = oracle.token_outputs(x[toks], ref_ids[toks], ref_w[toks], weights_of, res[toks])
    assert_close(host_f64(out[torch.from_numpy(toks).cuda()]), want, f"{name} fused-combine out")


def test_device_weight_generator_matches_host():
    """The device twin of the normal_bf16 stream gives the host generator's bits
    (it may differ only where the two math libraries round a transcendental
    differently right at a bf16 rounding boundary)."""
    n = 1 << 22
    for stream, offset in ((3, 0), (5, 123456789)):
        d = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        synth.normal_bf16_device(d, 0, stream, std=0.02, offset=offset)
        h = synth.normal_bf16(0, stream, (n,), std=0.02, offset=offset)
        mismatches = int(np.count_nonzero(host_u16(d) != h))
        assert mismatches <= 4, mismatches
