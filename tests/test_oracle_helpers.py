"""Pins of the oracle's helpers: the bf16 widening every float pin relies on,
and the per-layer counters of "Expert Coupling" Sec. II-B, Table I
(``layout_stats``).

Each check takes the function under test as an argument, so that the mutation
tests can run the same checks on planted mistakes.
"""
import math
import os
import struct
import json
from collections import Counter

import numpy as np
import pytest
import torch

import oracle
from test_oracle_layout import GOLDEN, expected_distinct_ranks, expected_same_rank_share, random_ids

ALL_BF16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


# ---- widen_bf16 ---------------------------------------------------------------------------
# The NaN patterns among the 65,536 make numpy's float32 -> float64 cast raise
# its "invalid value" warning; the NaNs themselves are what the checks compare.
NAN_CAST = pytest.mark.filterwarnings("ignore:invalid value encountered in cast:RuntimeWarning")

def check_widen_matches_torch(widen):
    """All 65,536 bit patterns against torch's own bfloat16 -> float64
    conversion: same NaN positions, same values elsewhere, same sign of zero."""
    got = np.asarray(widen(ALL_BF16), dtype=np.float64)
    ref = torch.from_numpy(ALL_BF16.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert got.shape == ref.shape
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def check_widen_matches_ieee_bytes(widen):
    """All patterns against the IEEE binary32 decoding of the pattern followed
    by sixteen zero bits (bf16 is the top half of a binary32), decoded by the
    struct module rather than by numpy."""
    got = np.asarray(widen(ALL_BF16), dtype=np.float64)
    for b in range(0, 1 << 16, 1):
        v = struct.unpack(">f", bytes([b >> 8, b & 0xFF, 0, 0]))[0]
        g = got[b]
        if math.isnan(v):
            assert math.isnan(g), hex(b)
        else:
            assert g == v and math.copysign(1.0, g) == math.copysign(1.0, v), hex(b)


HAND = [
    (0x3F80, 1.0),
    (0xC000, -2.0),
    (0x3F81, 1.0 + 2.0 ** -7),
    (0x4049, 3.140625),
    (0x0001, 2.0 ** -133),                       # smallest subnormal
    (0x0080, 2.0 ** -126),                       # smallest normal
    (0x7F7F, (2.0 - 2.0 ** -7) * 2.0 ** 127),    # largest finite
    (0x7F80, math.inf),
    (0xFF80, -math.inf),
    (0x0000, 0.0),
]


def check_widen_hand_values(widen):
    for bits, want in HAND:
        got = float(np.asarray(widen(np.array([bits], np.uint16)))[0])
        assert got == want, (hex(bits), got, want)
    nz = float(np.asarray(widen(np.array([0x8000], np.uint16)))[0])
    assert nz == 0.0 and math.copysign(1.0, nz) == -1.0, "0x8000 must widen to -0.0"
    for bits in (0x7FC0, 0xFFC1, 0x7F81):
        assert math.isnan(float(np.asarray(widen(np.array([bits], np.uint16)))[0])), hex(bits)


WIDEN_PINS = [check_widen_hand_values, check_widen_matches_torch, check_widen_matches_ieee_bytes]


@NAN_CAST
def test_widen_bf16_matches_torch_on_every_pattern():
    check_widen_matches_torch(oracle.widen_bf16)


@NAN_CAST
def test_widen_bf16_matches_the_ieee_decoding_of_every_pattern():
    check_widen_matches_ieee_bytes(oracle.widen_bf16)


@NAN_CAST
def test_widen_bf16_hand_values():
    check_widen_hand_values(oracle.widen_bf16)


def test_widen_bf16_keeps_the_shape():
    a = np.array([[0x3F80, 0x4000, 0x4040], [0xBF80, 0x0000, 0x8000]], np.uint16)
    assert np.array_equal(oracle.widen_bf16(a), [[1.0, 2.0, 3.0], [-1.0, 0.0, -0.0]])
    assert oracle.widen_bf16(a).dtype == np.float64


# ---- layout_stats (Expert Coupling, Sec. II-B, Table I) -----------------------------------

def stats_of(stats_fn, ids, placement, E, W):
    N, k = ids.shape
    return stats_fn(oracle.dispatch_layout(ids, placement, E, W), N, k, W)


def check_stats_worked_example(stats_fn):
    """The W = 3, top-2 example of the kernel-fusion page: every token's two
    experts sit on two ranks, so nothing merges and no token stays on one rank."""
    g = json.load(open(os.path.join(GOLDEN, "worked_routing_example.json")))
    ids = np.array([g["routing"][t] for t in g["tokens"]], np.int32)
    s = stats_of(stats_fn, ids, np.arange(g["E"]), g["E"], g["W"])
    assert s["rows"] == 6 and s["dedup_rows"] == 6
    assert s["ranks_per_token"] == 2.0
    assert s["same_rank_share"] == 0.0
    assert s["dedup_reduction"] == 0.0
    assert s["max_over_mean_load"] == 1.0


def check_stats_by_definition(stats_fn):
    """Each counter recomputed from its definition with Python sets and a
    Counter, on tie-free random routing under a permuted placement."""
    N, E, k, W = 300, 16, 3, 4
    ids = random_ids(N, E, k, seed=5)
    placement = np.random.default_rng(3).permutation(E)
    rank = {int(e): p // (E // W) for p, e in enumerate(placement)}
    per_token = [len({rank[int(e)] for e in ids[t]}) for t in range(N)]
    load = Counter(int(e) for e in ids.reshape(-1))
    s = stats_of(stats_fn, ids, placement, E, W)
    assert s["rows"] == N * k
    assert s["dedup_rows"] == sum(per_token)
    assert s["ranks_per_token"] == pytest.approx(sum(per_token) / N, abs=1e-12)
    assert s["same_rank_share"] == pytest.approx(sum(d == 1 for d in per_token) / N, abs=1e-12)
    assert s["dedup_reduction"] == pytest.approx(1 - sum(per_token) / (N * k), abs=1e-12)
    assert s["max_over_mean_load"] == pytest.approx(max(load.values()) / (N * k / E), abs=1e-12)


def check_stats_special_cases(stats_fn):
    """One rank: every token on one rank, d = 1.  One expert per rank: d = k,
    nothing merges (k > 1)."""
    N, E, k = 80, 8, 3
    ids = random_ids(N, E, k, seed=12)
    one = stats_of(stats_fn, ids, np.arange(E), E, 1)
    assert one["ranks_per_token"] == 1.0 and one["same_rank_share"] == 1.0
    assert one["dedup_reduction"] == pytest.approx(1 - 1 / k)
    per = stats_of(stats_fn, ids, np.arange(E), E, E)
    assert per["ranks_per_token"] == k and per["same_rank_share"] == 0.0
    assert per["dedup_reduction"] == 0.0


def check_stats_table1(stats_fn):
    """Table I's contiguous rows (E = 128): with iid routing the oracle's
    counters must sit within 4 sigma of the closed form, and within the
    table's rounding plus 4 sigma of the printed values."""
    g = json.load(open(os.path.join(GOLDEN, "table1_contiguous.json")))
    E, N = g["E"], 3000
    for row in g["rows"]:
        k, W = row["k"], row["EP"]
        ids = random_ids(N, E, k, seed=1000 + 10 * k + W)
        lay = oracle.dispatch_layout(ids, np.arange(E), E, W)
        s = stats_fn(lay, N, k, W)
        mu, p = expected_distinct_ranks(E, W, k), expected_same_rank_share(E, W, k)
        # the per-token count lies in [1, min(k, W)], so its standard deviation
        # is at most (min(k, W) - 1) / 2; sd bounds the standard error of the mean
        sd = max(0.5 * (min(k, W) - 1), 1e-9) / math.sqrt(N)
        sd_p = math.sqrt(max(p * (1 - p), 1.0 / N) / N)
        assert abs(s["ranks_per_token"] - mu) <= 4 * sd, (row, s)
        assert abs(s["ranks_per_token"] - row["gpus"]) <= 0.03 + 4 * sd, (row, s)
        assert abs(s["same_rank_share"] - p) <= 4 * sd_p, (row, s)
        assert abs(100 * s["same_rank_share"] - row["same_gpu_pct"]) <= 1.0 + 400 * sd_p, (row, s)
        assert abs(100 * s["dedup_reduction"] - row["dedup_pct"]) <= 1.0 + 400 * sd / k, (row, s)


STATS_PINS = [check_stats_worked_example, check_stats_by_definition, check_stats_special_cases,
              check_stats_table1]


@pytest.mark.parametrize("pin", STATS_PINS)
def test_layout_stats(pin):
    pin(oracle.layout_stats)
