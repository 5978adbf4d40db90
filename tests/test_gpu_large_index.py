"""A layer whose buffers hold more than 2^31 elements: y (and the plain
dispatched rows) span N*k*H = 65536*8*4352 = 2.28e9 bf16 values, so any row
offset computed in 32-bit arithmetic anywhere on the path would wrap.  Checked
against the oracle on the tokens of the highest rows of every expert segment
(the last ones reach the top of the index space), the first and last token and
a seeded sample; routing ids and the layout tables in full."""
import numpy as np
import pytest
import torch

import oracle
from combine_warp_top_gb300 import moe, synth
from gpu_util import assert_close, host_f64

pytestmark = pytest.mark.gpu

WL = synth.Workload("large_index", 65536, 4352, 16, 8, 256, 4)


def bf16_dev(a):
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()


@pytest.fixture(scope="module")
def inputs():
    return synth.make_logits(WL), synth.make_x(WL), synth.make_residual(WL)


@pytest.mark.parametrize("gemm,dedup", [("auto", False), ("single", False), ("auto", True)])
def test_layer_beyond_2_31_elements(inputs, gemm, dedup):
    wl = WL
    N, k, H = wl.N, wl.k, wl.H
    assert N * k * H > 2 ** 31
    shape = moe.Shape(N, H, wl.E, k, wl.W, wl.I, dedup=dedup, gemm=gemm)
    layer = moe.MoELayer(shape, synth.make_weight_device(wl, "gate"),
                         synth.make_weight_device(wl, "up"), synth.make_weight_device(wl, "down"))
    L, x, res = inputs
    out = layer.forward(torch.from_numpy(L).cuda(), bf16_dev(x), bf16_dev(res))
    torch.cuda.synchronize()
    layer.check_device_errors()
    ref_ids, ref_w = oracle.route(L, k)
    assert np.array_equal(layer.topk_ids.view(N, k).cpu().numpy(), ref_ids)
    ref = oracle.dispatch_layout(ref_ids, np.arange(wl.E), wl.E, wl.W)
    got = {n: t.cpu().numpy() for n, t in layer.layout.tensors.items()}
    for key in ("expert_counts", "expert_offsets", "row_token"):
        assert np.array_equal(got[key][:len(ref[key])], ref[key]), key
    assert np.array_equal(got["pair_row"].reshape(N, k), ref["pair_row"])
    if dedup:
        assert int(got["n_dedup_rows"][0]) == ref["n_dedup_rows"]
    # tokens of the last two rows of every expert, the ends, and a sample
    off, cnt = ref["expert_offsets"], ref["expert_counts"]
    tail_rows = [int(off[e]) + int(cnt[e]) - d for e in range(wl.E) for d in (1, 2)
                 if cnt[e] >= d]
    rng = np.random.default_rng(5)
    toks = np.unique(np.concatenate([ref["row_token"][tail_rows], [0, N - 1],
                                     rng.choice(N, size=16, replace=False)])).astype(np.int64)

    def weights_of(e):
        return tuple(synth.make_weight(wl, m, experts=[e])[0] for m in ("gate", "up", "down"))

    want, y_want = oracle.token_outputs(x[toks], ref_ids[toks], ref_w[toks], weights_of, res[toks])
    assert_close(host_f64(out[torch.from_numpy(toks).cuda()]), want, "out")
    pr = ref["pair_row"][toks].reshape(-1).astype(np.int64)
    assert int(pr.max()) * H > 2 ** 31  # the checked rows reach past 2^31 elements
    assert_close(host_f64(layer.y[torch.from_numpy(pr).cuda()]), y_want.reshape(-1, H), "y rows")
