"""Runs the stages of a benchmark workload that need no expert weights -- route,
dispatch layout and (plain form) dispatch -- a few times through the C ABI, so
that a profiler can capture their kernels on the workload's own shape with only
its logits and token rows on the device.  With --layer it runs the whole layer
instead (random-init expert weights, packed), so that the expert FFN's kernels
can be captured too; the shape options turn the workload into a smaller or
differently shaped case.  Nothing is timed here.

    python -m combine_warp_top_gb300.profile_stages --workload deepseek_v3 --reps 3
    python -m combine_warp_top_gb300.profile_stages --workload tiny --layer --gemm fused \\
        --tokens 16384 --hidden 256 --experts 16 --topk 4 --inter 1408 --ranks 4
"""
from __future__ import annotations

import argparse
import dataclasses

import numpy as np
import torch

from . import moe, synth


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--workload", default="deepseek_v3", choices=sorted(synth.WORKLOADS))
    p.add_argument("--reps", type=int, default=3)
    p.add_argument("--no-dispatch", action="store_true", help="route and layout only")
    p.add_argument("--layer", action="store_true", help="the whole layer (moe_layer_forward)")
    p.add_argument("--gemm", default="auto", choices=sorted(moe.GEMM_KERNELS))
    for name, field in (("tokens", "N"), ("hidden", "H"), ("experts", "E"), ("topk", "k"),
                        ("inter", "I"), ("ranks", "W")):
        p.add_argument(f"--{name}", type=int, default=None, help=f"override {field}")
    args = p.parse_args(argv)

    wl = synth.WORKLOADS[args.workload]
    changes = {f: getattr(args, n) for n, f in (("tokens", "N"), ("hidden", "H"),
                                                 ("experts", "E"), ("topk", "k"),
                                                 ("inter", "I"), ("ranks", "W"))
               if getattr(args, n) is not None}
    if changes:
        wl = dataclasses.replace(wl, name=f"{wl.name}_custom", **changes)
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=wl.dedup, gemm=args.gemm)
    logits = torch.from_numpy(synth.make_logits(wl)).cuda()
    placement = (None if wl.placement == "contiguous" or changes
                 else torch.from_numpy(synth.make_placement(wl)).cuda())
    if args.layer:
        x = torch.from_numpy(synth.make_x(wl).view(np.int16)).view(torch.bfloat16).cuda()
        w = [synth.make_weight_device(wl, m) for m in ("gate", "up", "down")]
        layer = moe.MoELayer(shape, *w, placement)
        del w
        for _ in range(args.reps):
            layer.forward(logits, x, None)
        torch.cuda.synchronize()
        layer.check_device_errors()
        print(f"{wl.name} N={wl.N} H={wl.H} E={wl.E} k={wl.k} I={wl.I} W={wl.W}: "
              f"{args.reps} x layer ok ({'fused FFN' if layer.fused_ffn else 'two GEMMs'})")
        return
    ids = torch.empty(wl.N * wl.k, dtype=torch.int32, device="cuda")
    w = torch.empty(wl.N * wl.k, dtype=torch.float32, device="cuda")
    layout, ws = moe.Layout(shape), moe.workspace(shape)
    x = xd = None
    if not args.no_dispatch:
        x = torch.from_numpy(synth.make_x(wl).view(np.int16)).view(torch.bfloat16).cuda()
        xd = torch.empty(moe._rows_d(shape), wl.H, dtype=torch.bfloat16, device="cuda")
    for _ in range(args.reps):
        moe.moe_route(logits, shape, ids, w)
        moe.moe_dispatch_layout(ids, placement, shape, layout, ws)
        if xd is not None:
            moe.moe_dispatch(x, layout, shape, xd)
    torch.cuda.synchronize()
    status = moe.moe_get_error(ws)
    if status != 0:
        raise SystemExit(f"device error: {moe.moe_status_str(status)}")
    print(f"{args.workload}: {args.reps} x (route, dispatch layout"
          f"{'' if xd is None else ', dispatch'}) ok")


if __name__ == "__main__":
    main()
