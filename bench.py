#!/usr/bin/env python
"""Throughput of the MoE layer forward pass on GB300.

One step = one pass of the whole path (route, dispatch layout, dispatch,
[dedup expansion], gate/up GEMM + SwiGLU, down GEMM, combine + residual) over
one batch of synthetic tokens, with inputs and expert weights resident in HBM.
The default workload is the DeepSeek-V3-shaped layer (N=4096 tokens, H=7168,
E=256 experts, top-8, SwiGLU width 2048, W=8 ranks); its 22.5 GB of expert
weights are read every step, far more than the 129 MB L2, so no L2 flush is
needed between steps.

Prints one JSON line.  --impl reference times the CPU oracle instead (the
plain float64 restatement of the layer) on a bounded sample of the same
workload.  Under torchrun (N > 1) every rank runs its own replica of the layer
on its own tokens (weak scaling, no collective on the data path); the reported
time is the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import datetime as dt
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (1 GB300); dispatch/combine HBM GB/s; grouped-GEMM TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="deepseek_v3")
    p.add_argument("--tokens", type=int, default=None, help="override N (profiling cases)")
    p.add_argument("--experts", type=int, default=None, help="override E (profiling cases)")
    p.add_argument("--dedup", choices=["auto", "on", "off"], default="auto")
    p.add_argument("--weights", choices=["packed", "row_major"], default="packed",
                   help="expert weights as moe_pack_weights' tile-contiguous copy (packed once "
                        "before timing) or in nn.Linear layout")
    p.add_argument("--gemm", choices=["auto", "single", "pair", "fused"], default="auto",
                   help="grouped-GEMM kernel (the shape's gemm field)")
    p.add_argument("--placement-search", action="store_true",
                   help="place experts by the co-selection search before timing the layer")
    p.add_argument("--shared-expert", type=int, default=0, metavar="I_S",
                   help="add a shared expert of SwiGLU width I_S to every step")
    p.add_argument("--microbatch", type=int, default=0, metavar="T",
                   help="run the step as a two-stream pipeline of T-token microbatches")
    p.add_argument("--fuse-combine", action="store_true",
                   help="down GEMM with the combine in its epilogue (moe_ffn_down_combine)")
    p.add_argument("--eager", action="store_true",
                   help="launch every step from Python instead of replaying a captured CUDA graph")
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--others", default="auto",
                   help="workloads measured after the headline one: a comma list, 'none', or "
                        "'auto' (the five other benchmark workloads when the default "
                        "DeepSeek-V3 layer runs on one GPU without options)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--oracle-worker", default=None, help=argparse.SUPPRESS)
    return p.parse_args(argv)


# ---------------------------------------------------------------------------- workload

def workload(args):
    from combine_warp_top_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    changes = {}
    if args.tokens is not None:
        changes["N"] = args.tokens
    if args.experts is not None:
        changes["E"] = args.experts
        changes["W"] = min(wl.W, args.experts)
    if args.dedup != "auto":
        changes["dedup"] = args.dedup == "on"
    if changes:
        import dataclasses
        wl = dataclasses.replace(wl, name=wl.name + "_" + "_".join(f"{k}{v}" for k, v in changes.items()),
                                 **changes)
    return wl


def algorithmic(wl, R_d, fused_dispatch=False):
    """Bytes each stage must move and flops it must do (bf16 activations and
    weights, fp32 logits and weights of the router).  The gate/up GEMM reads
    its A rows once from wherever they live: the dispatched rows (plain), the
    dedup rows it expands itself (dedup), or x itself when it also does the
    dispatch (fused_dispatch)."""
    N, H, E, k, I, W = wl.N, wl.H, wl.E, wl.k, wl.I, wl.W
    R = N * k
    rows_d = R_d if wl.dedup else R
    a_rows = R_d if wl.dedup else (N if fused_dispatch else R)
    st = {
        "route": dict(bytes=N * E * 4 + R * 8),
        "layout": dict(bytes=2 * R * 4 + (5 if wl.dedup else 2) * R * 4),
        "dispatch": dict(bytes=N * H * 2 + rows_d * H * 2),
        "gate_up": dict(bytes=2 * E * I * H * 2 + a_rows * H * 2 + R * I * 2, flops=4 * R * H * I),
        "down": dict(bytes=E * H * I * 2 + R * I * 2 + R * H * 2, flops=2 * R * H * I),
        # both GEMMs in one kernel with h on chip: weights, the rows once, y out
        "ffn": dict(bytes=3 * E * I * H * 2 + a_rows * H * 2 + R * H * 2, flops=6 * R * H * I),
        # dedup: the partial rows stay in registers (one-pass dedup combine)
        "combine": dict(bytes=R * H * 2 + 2 * N * H * 2 + R * 8),
        # down GEMM with the combine in its epilogue: weights, h in, residual
        # in, out; y never leaves the SM
        "down_combine": dict(bytes=E * H * I * 2 + R * I * 2 + 2 * N * H * 2 + R * 8,
                             flops=2 * R * H * I),
    }
    return st


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


TRAFFIC_SOURCES = ("combine_warp_top_gb300/csrc/grouped_gemm.cu",
                   "combine_warp_top_gb300/csrc/grouped_gemm_2sm.cu",
                   "combine_warp_top_gb300/csrc/ptx.cuh")


def code_lines(text):
    """The lines of a C++/CUDA source that are code: // comments, trailing
    blanks and empty lines removed (the sources hold no '//' inside strings)."""
    out = []
    for line in text.splitlines():
        code = line.split("//", 1)[0].rstrip()
        if code:
            out.append(code)
    return "\n".join(out)


def sources_digest():
    """sha256 prefix over the code of the grouped-GEMM sources (both kernels and
    their PTX wrappers, comments ignored): a recorded DRAM traffic figure holds
    only for this code."""
    import hashlib
    h = hashlib.sha256()
    for rel in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel)) as f:
            h.update(code_lines(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(wl):
    """DRAM bytes (read + write) of one gate/up GEMM launch of this workload,
    from the committed ncu capture (profiles/gemm_traffic.json: one full-size
    capture per workload); None if the capture does not cover this workload
    or the GEMM sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("sources_sha256_prefix") != sources_digest():
        return None
    entry = rec.get("gate_up", {}).get(wl.name)
    return None if entry is None else entry["dram_bytes"]


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ["timestamp", "index", "clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(1.0)  # nvidia-smi needs a moment before its first sample

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                ts = dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 <= r[0] <= self.t1]
        window = "timed region"
        if len(inside) < 3:
            inside = [r for r in rows if self.t0 - 0.5 <= r[0] <= self.t1 + 0.5]
            window = "timed region +-0.5 s"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median([r[1] for r in inside]) if inside else None,
                "sm_max_mhz": max((r[2] for r in inside), default=None),
                "reasons": reasons, "samples": len(inside), "window": window}


# ---------------------------------------------------------------------------- oracle timing

COMBINE_SAMPLE_TOKENS = 1024


def oracle_worker(spec):
    """Times the CPU oracle's steps of one layer step of the workload, in its
    own process (the BLAS thread count is set by the caller's environment).

    Sample, per step:
      * route, dispatch layout and dispatch (dedup: the dedup rows and their
        expansion) over all N tokens;
      * the expert FFN: oracle.swiglu_mlp, the oracle's per-expert step, on the
        rows this routing gives each of ``experts_per_step`` seeded experts
        (their weights generated and widened before the timer starts), scaled
        to all R = N*k rows by the share of rows the sampled experts hold;
      * the combine (plain: oracle.combine; dedup: oracle.combine_dedup) over
        the first min(N, 1024) tokens, scaled to N.
    Successive steps take successive experts of one seeded permutation."""
    import numpy as np

    import oracle
    from combine_warp_top_gb300 import synth
    args = parse_args(spec["argv"])
    wl = workload(args)
    rng = np.random.default_rng(spec.get("seed", 0))
    L = synth.make_logits(wl)
    x = synth.make_x(wl)
    res = synth.make_residual(wl)
    placement = synth.make_placement(wl)
    N, k, H = wl.N, wl.k, wl.H
    R = N * k
    # untimed: which experts hold rows under this routing (the sample's pool)
    ids0, _ = oracle.route(L, k)
    counts0 = np.bincount(ids0.reshape(-1), minlength=wl.E)
    pool = rng.permutation(np.nonzero(counts0)[0])
    n_sub = min(N, COMBINE_SAMPLE_TOKENS)
    y_rows = rng.standard_normal((R, H)) if n_sub == N else None
    steps, nxt = [], 0
    for _ in range(spec["steps"]):
        experts = [int(pool[(nxt + i) % len(pool)]) for i in range(spec["experts_per_step"])]
        experts = sorted(set(experts))
        nxt += spec["experts_per_step"]
        weights = {e: tuple(oracle.widen_bf16(synth.make_weight(wl, m, experts=[e])[0])
                            for m in ("gate", "up", "down")) for e in experts}
        t = {}
        c = time.perf_counter()
        ids, w = oracle.route(L, k)
        t["route"] = time.perf_counter() - c
        c = time.perf_counter()
        lay = oracle.dispatch_layout(ids, placement, wl.E, wl.W)
        t["layout"] = time.perf_counter() - c
        c = time.perf_counter()
        if wl.dedup:
            xd = oracle.expand(oracle.dispatch_dedup(x, lay["dedup_row_token"]), lay["expand_src"])
        else:
            xd = oracle.dispatch(x, lay["row_token"])
        t["dispatch"] = time.perf_counter() - c
        rows, ffn = 0, 0.0
        for e in experts:
            a, n = int(lay["expert_offsets"][e]), int(lay["expert_counts"][e])
            c = time.perf_counter()
            oracle.swiglu_mlp(oracle.widen_bf16(xd[a:a + n]), *weights[e])
            ffn += time.perf_counter() - c
            rows += n
        t["ffn"] = ffn * R / max(rows, 1)
        # combine over the first n_sub tokens: their k rows, compacted
        pr = lay["pair_row"][:n_sub]
        y_sub = y_rows[pr.reshape(-1)] if y_rows is not None else \
            rng.standard_normal((n_sub * k, H))
        pr_sub = np.arange(n_sub * k).reshape(n_sub, k)
        c = time.perf_counter()
        if wl.dedup:
            d = lay["pair_dedup_row"][:n_sub]
            uniq, dd = np.unique(d, return_inverse=True)
            oracle.combine_dedup(y_sub, w[:n_sub], pr_sub, dd.reshape(n_sub, k), len(uniq),
                                 res[:n_sub])
        else:
            oracle.combine(y_sub, w[:n_sub], pr_sub, res[:n_sub])
        t["combine"] = (time.perf_counter() - c) * N / n_sub
        total = sum(t.values())
        steps.append({"seconds": total, "tokens": N, "stage_s": t, "experts": experts,
                      "rows_sampled": rows})
    return {"steps": steps, "threads": spec["threads"], "n_sub": n_sub}


def run_oracle(argv, threads, steps=1, experts_per_step=4, seed=0):
    """The oracle worker in a subprocess whose BLAS and OpenMP pools have
    `threads` threads."""
    n = str(threads)
    env = dict(os.environ, OMP_NUM_THREADS=n, OPENBLAS_NUM_THREADS=n, MKL_NUM_THREADS=n)
    spec = json.dumps({"argv": argv, "steps": steps, "experts_per_step": experts_per_step,
                       "seed": seed, "threads": threads})
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-worker", spec],
                       capture_output=True, text=True, env=env, cwd=ROOT)
    if r.returncode != 0:
        raise RuntimeError("oracle worker failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def oracle_sample_text(wl, experts_per_step, steps, n_sub):
    return (f"each step: route, dispatch layout and dispatch of all {wl.N} tokens of the "
            f"{wl.name} workload; the expert FFN (oracle.swiglu_mlp, weights widened before "
            f"timing) on the rows of {experts_per_step} seeded experts, scaled to all "
            f"{wl.N * wl.k} rows by the rows they hold; the combine over {n_sub} tokens, scaled "
            f"to {wl.N}; float64 numpy; {steps} step(s)")


def cpu_baseline(argv, wl):
    """The oracle timed with every host core and with one (bounded samples)."""
    ncpu = os.cpu_count() or 1
    runs = {}
    for threads, experts in ((ncpu, 8), (1, 2)):
        r = run_oracle(argv, threads, steps=1, experts_per_step=experts)
        st = r["steps"][0]
        runs[threads] = (st, r["n_sub"], experts)
    st, n_sub, experts = runs[ncpu]
    st1, n_sub1, experts1 = runs[1]
    return {
        "value": round(st["tokens"] / st["seconds"], 3), "unit": "tokens/s", "cores": ncpu,
        "kind": "oracle",
        "sample": oracle_sample_text(wl, experts, 1, n_sub) +
                  f"; {ncpu} threads in the BLAS calls (the other steps are single-threaded numpy)",
        "stage_s": {k: round(v, 4) for k, v in st["stage_s"].items()},
        "one_core": {"value": round(st1["tokens"] / st1["seconds"], 3), "unit": "tokens/s",
                     "cores": 1, "sample": oracle_sample_text(wl, experts1, 1, n_sub1),
                     "stage_s": {k: round(v, 4) for k, v in st1["stage_s"].items()}},
    }


def strip_args(argv):
    keep, skip = [], False
    for a in argv:
        if skip:
            skip = False
            continue
        if a in ("--impl", "--gpus", "--steps", "--warmup", "--e2e-steps", "--others"):
            skip = True
            continue
        if a.startswith("--impl=") or a == "--no-cpu-baseline":
            continue
        keep.append(a)
    return keep


# ---------------------------------------------------------------------------- distributed

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, local):
    import torch
    import torch.distributed as dist
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return dist


def max_over_ranks(value, world):
    """Largest value over the ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    if world == 1:
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    import torch.distributed as dist
    if world > 1:
        dist.barrier()


# ---------------------------------------------------------------------------- placement search

def placement_search(wl, shape, logits_d, repeats=20):
    """Correlated placement from this batch's routing: co-selection counts on
    the GPU (timed with CUDA events), best-swap search on the host (timed by
    wall clock), and the dedup rows under contiguous, planted and searched
    placement."""
    import torch

    from combine_warp_top_gb300 import moe, synth
    ids = torch.empty(wl.N * wl.k, dtype=torch.int32, device="cuda")
    w = torch.empty(wl.N * wl.k, dtype=torch.float32, device="cuda")
    moe.moe_route(logits_d, shape, ids, w)
    ws = moe.workspace(shape)
    W = torch.empty(wl.E, wl.E, dtype=torch.int32, device="cuda")
    moe.moe_coselection(ids, shape, W, ws)  # warm-up
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(repeats):
        moe.moe_coselection(ids, shape, W, ws)
    e1.record()
    torch.cuda.synchronize()
    cos_ms = e0.elapsed_time(e1) / repeats
    W_h = W.cpu()
    t0 = time.perf_counter()
    placement, swaps = moe.moe_placement_search(W_h, wl.W)
    search_ms = (time.perf_counter() - t0) * 1e3

    def rows(pl):
        dshape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=True)
        lay = moe.Layout(dshape)
        moe.moe_dispatch_layout(ids, None if pl is None else pl.cuda(), dshape, lay, moe.workspace(dshape))
        torch.cuda.synchronize()
        return int(lay["n_dedup_rows"].item())

    out = {"coselection_ms": round(cos_ms, 4),
           "coselection_pairs_per_s": round(wl.N * wl.k * wl.k / cos_ms * 1e3, 1),
           "search_ms": round(search_ms, 2), "swaps": swaps,
           "dedup_rows_contiguous": rows(None), "dedup_rows_searched": rows(placement),
           "placement": placement}
    if wl.logits == "hot_pairs":
        out["dedup_rows_planted"] = rows(torch.from_numpy(synth.make_placement(
            synth.WORKLOADS["correlated_placed"])))
    return out


# ---------------------------------------------------------------------------- our arm

OTHER_WORKLOADS = ("tiny", "mixtral", "correlated_contiguous", "correlated_placed", "skewed")


def measure(args, wl, world, rank, headline=True):
    """Builds the layer of workload `wl`, times K steps (after W warm-up
    steps) and returns its figures.  headline=False skips the end-to-end run,
    the placement search and the microbatch / fused-combine / shared-expert
    options (the other benchmark workloads are measured as plain layers)."""
    import numpy as np
    import torch

    from combine_warp_top_gb300 import moe, synth

    seed = rank  # every rank has its own tokens; weights are the same layer
    shape = moe.Shape(wl.N, wl.H, wl.E, wl.k, wl.W, wl.I, dedup=wl.dedup, gemm=args.gemm)

    w_gate = synth.make_weight_device(wl, "gate")
    w_up = synth.make_weight_device(wl, "up")
    w_down = synth.make_weight_device(wl, "down")
    placement = synth.make_placement(wl)
    placement_d = None if wl.placement == "contiguous" else torch.from_numpy(placement).cuda()
    L_h = torch.from_numpy(synth.make_logits(wl, seed)).pin_memory()
    search = None
    if headline and args.placement_search:
        search = placement_search(wl, shape, L_h.cuda())
        placement_d = search.pop("placement").cuda()
    shared = None
    if headline and args.shared_expert:
        I_s = args.shared_expert
        shared = tuple(synth.normal_bf16_device(
            torch.empty(*shp, dtype=torch.bfloat16, device="cuda"), 0, stream_id, std=0.02)
            for stream_id, shp in ((103, (I_s, wl.H)), (104, (I_s, wl.H)), (105, (wl.H, I_s))))
    fuse_combine = headline and args.fuse_combine
    microbatch = args.microbatch if headline else 0
    if fuse_combine and (microbatch or shared is not None):
        raise SystemExit("--fuse-combine runs the plain layer: no --microbatch, no --shared-expert")
    pack = args.weights == "packed"
    layer = moe.MoELayer(shape, w_gate, w_up, w_down, placement_d, shared=shared,
                         fuse_combine=fuse_combine, pack=pack)
    if pack and not microbatch:
        # the layer holds its packed copy; the row-major matrices can go
        w_gate = w_up = w_down = None
        torch.cuda.empty_cache()

    x_h = torch.from_numpy(synth.make_x(wl, seed).view(np.int16)).view(torch.bfloat16).pin_memory()
    r_h = torch.from_numpy(synth.make_residual(wl, seed).view(np.int16)).view(torch.bfloat16).pin_memory()
    out_h = torch.empty(wl.N, wl.H, dtype=torch.bfloat16).pin_memory()
    L_d, x_d, r_d = L_h.cuda(), x_h.cuda(), r_h.cuda()
    torch.cuda.synchronize()

    rows = dispatch_rows(wl, shape, L_d, placement_d)

    stream = torch.cuda.current_stream()
    pipe = None
    if microbatch:
        pipe = moe.MicrobatchPipeline(shape, w_gate, w_up, w_down, placement_d,
                                      microbatch=microbatch, shared=shared, pack=pack)
    runner = pipe if pipe is not None else layer
    n_mb = len(pipe.chunks()) if pipe is not None else 0

    use_graph = pipe is None and not args.eager
    alone_ms = {}

    def step(i):
        if pipe is None:
            layer.forward_stages(L_d, x_d, r_d, events=ev[i])
        else:
            pipe.forward(L_d, x_d, r_d, out=layer.out, gemm_events=gev[i])

    stages = layer.stage_names()
    dom = dominant_stage(layer)
    # external events: inside a captured graph they become timing nodes.  The
    # headline's timed graph carries them around the dominant stage (gate/up)
    # only: a pair around every stage of every step cost 0.5-1.8% of the step
    # on GB300.  The other workloads' timed graphs carry none (one pair per
    # step added 10 us to the 26 us tiny step).  Stages without live events are
    # timed by a second, instrumented replay after the timed region
    # (instrumented_stage_ms).
    mk = lambda: (torch.cuda.Event(enable_timing=True, external=use_graph),  # noqa: E731
                  torch.cuda.Event(enable_timing=True, external=use_graph))
    timed_stages = ([dom] if headline else []) if use_graph else stages
    ev = [{s: mk() for s in timed_stages} for _ in range(args.steps)] if pipe is None else None
    gev = [[mk() for _ in range(n_mb)] for _ in range(args.steps)] if pipe is not None else None
    for i in range(args.warmup):
        step(i % args.steps)
    torch.cuda.synchronize()
    runner.check_device_errors()
    graph = None
    if use_graph:
        # the whole timed loop as one CUDA graph: K steps of the same kernels,
        # with the per-stage timing events recorded by graph nodes
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(args.steps):
                step(i)
        graph.replay()  # untimed: the graph's first launch uploads it
        torch.cuda.synchronize()
        runner.check_device_errors()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t0")
    t_start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            step(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t1")
    barrier(world)
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    clocks = sampler.stop() if sampler else None
    runner.check_device_errors()
    if pipe is None:
        stage_ms = {s: statistics.mean(e[s][0].elapsed_time(e[s][1]) for e in ev)
                    for s in timed_stages}
        if use_graph:
            # every stage, from one replay of the same K steps with timing
            # nodes around each; the headline's gate/up keeps the timed
            # region's figure
            full = instrumented_stage_ms(layer, L_d, x_d, r_d, stages, args.steps)
            stage_ms = {s: stage_ms.get(s, full[s]) for s in stages}
            alone_ms = stage_alone_ms(layer, L_d, x_d, r_d, stages, args.steps)
            runner.check_device_errors()
    else:
        # gate/up (or fused FFN) launches of all microbatches of a step, on the
        # GEMM stream
        stage_ms = {dom: statistics.mean(sum(a.elapsed_time(b) for a, b in g) for g in gev)}
        stages = [dom]

    e2e = None
    if headline:
        # end to end through the public host-buffer API: every step copies its
        # inputs from pinned host memory and its output back, overlapped with
        # the neighbouring steps' compute (moe.HostPipeline)
        # 50 steps by default whatever K is: a few hundred ms of host-link
        # traffic, long enough that the host's scheduling jitter averages out
        e2e_steps = args.e2e_steps or 50
        host = moe.HostPipeline(runner, with_residual=True)
        batches = [(L_h, x_h, r_h, out_h)] * e2e_steps
        host.run(batches[:4])
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        host.run(batches)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
        runner.check_device_errors()
        e2e = {"value": round(wl.N * e2e_steps * world / (e2e_ms / 1e3), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": wl.N * wl.E * 4 + 2 * wl.N * wl.H * 2,
               "d2h_bytes_per_step": wl.N * wl.H * 2, "steps": e2e_steps}

    pk, pk_src = peaks()
    alg = algorithmic(wl, rows["dedup"], layer.fused_dispatch)
    if shared is not None:
        I_s = args.shared_expert
        alg["shared"] = dict(bytes=3 * I_s * wl.H * 2 + 2 * wl.N * wl.H * 2 + 2 * wl.N * I_s * 2,
                             flops=6 * wl.N * wl.H * I_s)
        alg["combine"]["bytes"] += wl.N * wl.H * 2
    ridge = pk["bf16_tflops_sustained"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    stage_report = {}
    for s in stages:
        ms = stage_ms[s]
        d = {"ms": round(ms, 4), "GB/s": round(alg[s]["bytes"] / ms / 1e6, 1)}
        d["hbm_frac"] = round(d["GB/s"] / pk["hbm_gbs"], 3)
        if "flops" in alg[s]:
            d["TFLOP/s"] = round(alg[s]["flops"] / ms / 1e9, 1)
            d["tensor_frac"] = round(d["TFLOP/s"] / pk["bf16_tflops_sustained"], 3)
            d["bound"] = "tensor" if alg[s]["flops"] / alg[s]["bytes"] > ridge else "hbm"
        else:
            d["bound"] = "hbm"
        if s in alone_ms:
            a_ms = alone_ms[s]
            d["alone_ms"] = round(a_ms, 4)
            d["alone_hbm_frac"] = round(alg[s]["bytes"] / a_ms / 1e6 / pk["hbm_gbs"], 3)
            if "flops" in alg[s]:
                d["alone_tensor_frac"] = round(alg[s]["flops"] / a_ms / 1e9 /
                                               pk["bf16_tflops_sustained"], 3)
        stage_report[s] = d

    roof = roofline(wl, alg, stage_ms, pk, pk_src, ridge, layer, pipe, n_mb)
    what = "fused FFN" if dom == "ffn" else "gate/up"
    roof["timed"] = (f"CUDA events around every {what} launch of the timed region"
                     if dom in timed_stages or pipe is not None else
                     f"CUDA events around every {what} launch of an instrumented replay of the "
                     "same K steps (this workload's timed region carries no timing node)")
    res = {
        "value": round(wl.N * args.steps * world / (elapsed_ms / 1e3), 1),
        "ms_per_step": round(elapsed_ms / args.steps, 4),
        "roofline": roof, "stages": stage_report, "clocks": clocks, "dispatch_rows": rows,
        "gpu_launches": runner.kernel_launches_per_step() * args.steps,
        "graph": graph is not None, "e2e": e2e, "search": search,
    }
    del graph, layer, pipe, runner, w_gate, w_up, w_down
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def dispatch_rows(wl, shape, L_d, placement_d):
    """Rows the plain and the deduplicating dispatcher send for this routing,
    with the per-layer counters of "Expert Coupling" Table I, from the
    library's own routing and layout tables (not timed)."""
    import numpy as np
    import torch

    from combine_warp_top_gb300 import moe
    dshape = dataclasses.replace(shape, dedup=True)
    ids = torch.empty(wl.N * wl.k, dtype=torch.int32, device="cuda")
    w = torch.empty(wl.N * wl.k, dtype=torch.float32, device="cuda")
    dlay, dws = moe.Layout(dshape), moe.workspace(dshape)
    moe.moe_route(L_d, shape, ids, w)
    moe.moe_dispatch_layout(ids, placement_d, dshape, dlay, dws)
    torch.cuda.synchronize()
    R, R_d = wl.N * wl.k, int(dlay["n_dedup_rows"].item())
    counts = dlay["expert_counts"].cpu().numpy()
    # distinct ranks of each token = its dedup rows
    per_token = np.bincount(dlay["dedup_row_token"][:R_d].cpu().numpy(), minlength=wl.N)
    return {"plain": R, "dedup": R_d, "dedup_reduction": round(1 - R_d / R, 4),
            "ranks_per_token": round(R_d / wl.N, 4),
            "same_rank_share": round(float(np.mean(per_token == 1)), 4),
            "max_over_mean_expert_load": round(float(counts.max() / counts.mean()), 3)}


def dominant_stage(layer):
    """The stage of the layer's dominant kernel: the gate/up GEMM, or the fused
    expert FFN where the layer runs both GEMMs as one kernel."""
    return "ffn" if layer.fused_ffn else "gate_up"


def roofline(wl, alg, stage_ms, pk, pk_src, ridge, layer, pipe, n_mb):
    """The roofline object of the dominant kernel (dominant_stage)."""
    dom = dominant_stage(layer)
    a = alg[dom]
    if a["flops"] / a["bytes"] > ridge:
        achieved = a["flops"] / stage_ms[dom] / 1e9
        roof = {"bound": "tensor", "achieved": round(achieved, 1),
                "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s"}
    else:
        achieved = a["bytes"] / stage_ms[dom] / 1e6
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 3)
    roof["traffic"] = recorded_traffic(wl) if dom == "gate_up" else None
    if roof["frac"] > 1.0:
        roof["note"] = ("above 1: the peak is a copy probe (half its bytes writes); this kernel "
                        "mostly reads, and its DRAM traffic is at least its algorithmic bytes, "
                        "so no L2 hit inflates the figure")
    if dom == "ffn":
        roof["kernel"] = ("fused_ffn_kernel (moe_ffn_fused: gate/up, SwiGLU and down in one "
                          "kernel, h kept on chip, rows gathered by its own warps)")
    elif wl.dedup:
        roof["kernel"] = ("grouped_gemm_kernel<SwiGLU, gathered rows> (moe_ffn_gate_up_gather: "
                          "the dedup expansion done by the GEMM's gather warps)")
    elif layer.fused_dispatch:
        roof["kernel"] = ("grouped_gemm_kernel<SwiGLU, gathered rows> (moe_ffn_gate_up_gather: "
                          "the dispatch copy done by the GEMM's gather warps)")
    else:
        roof["kernel"] = "grouped_gemm_kernel<SwiGLU> or its CTA-pair form (moe_ffn_gate_up)"
    if pipe is not None:
        roof["kernel"] += f", summed over the {n_mb} microbatches of a step"
    peak_key = "bf16_tflops_sustained" if roof["unit"] == "TFLOP/s" else "hbm_gbs"
    roof["peak_source"] = f"{pk_src} ({peak_key})"
    roof["algorithmic_per_launch"] = {"bytes": a["bytes"], "flops": a["flops"]}
    return roof


def workload_config(wl):
    return {"workload": wl.name, "N": wl.N, "H": wl.H, "E": wl.E, "k": wl.k, "I": wl.I,
            "W": wl.W, "dedup": wl.dedup, "placement": wl.placement}


def l2_note(wl):
    wbytes = 3 * wl.E * wl.H * wl.I * 2
    if wbytes > 129e6:
        return f"no flush: {wbytes / 1e9:.2f} GB of expert weights read per step, larger than the 129 MB L2"
    return (f"no flush: the {wbytes / 1e6:.1f} MB of weights fit in L2 and stay there from step to "
            f"step (a latency-bound case)")


def run_ours(args):
    world, rank, local = dist_info()
    dist_init(world, local)
    import torch
    torch.cuda.set_device(local)
    wl = workload(args)
    r = measure(args, wl, world, rank, headline=True)
    others = []
    if args.others == "auto":
        default = (args.workload == "deepseek_v3" and args.tokens is None and args.experts is None
                   and args.dedup == "auto" and not (args.microbatch or args.fuse_combine or
                                                     args.shared_expert or args.placement_search))
        others = list(OTHER_WORKLOADS) if default and world == 1 else []
    elif args.others != "none":
        others = [w for w in args.others.split(",") if w]
    extra = {}
    for name in others:
        from combine_warp_top_gb300 import synth
        o = measure(args, synth.WORKLOADS[name], world, rank, headline=False)
        extra[name] = {"value": o["value"], "unit": "tokens/s", "ms_per_step": o["ms_per_step"],
                       "config": workload_config(synth.WORKLOADS[name]),
                       "roofline": {k: o["roofline"][k] for k in ("bound", "achieved", "peak",
                                                                   "unit", "frac", "traffic")},
                       "stages": o["stages"], "dispatch_rows": o["dispatch_rows"],
                       "gpu_launches": o["gpu_launches"], "clocks": o["clocks"]}
    if rank != 0:
        return None
    cfg = workload_config(wl)
    cfg.update({
        "shared_expert_I": args.shared_expert or None,
        "fused_combine": bool(args.fuse_combine),
        "microbatch": args.microbatch or None,
        "gemm": args.gemm,
        "weights": (("packed once before timing (moe_pack_weights: every 64-deep slice of "
                     "a 256-row weight tile contiguous)") if args.weights == "packed"
                    else "row-major (nn.Linear layout)"),
        "launch": ("one CUDA graph of the K timed steps, timing nodes around gate/up only; "
                   "the other stages' times from a second, instrumented replay of the K steps")
                  if r["graph"] else "eager, one C call per stage",
        "parallelism": f"{world} independent replicas" if world > 1 else "1 GPU",
        "l2": l2_note(wl)})
    line = {
        "metric": METRIC,
        "value": r["value"],
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": r["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64/Box-Muller; random-init expert weights)",
        "config": cfg,
        "roofline": r["roofline"],
        "e2e": r["e2e"],
        "gpu_launches": r["gpu_launches"],
        "clocks": r["clocks"],
        "stages": r["stages"],
        "dispatch_rows": r["dispatch_rows"],
    }
    if r["search"] is not None:
        line["placement_search"] = r["search"]
    if extra:
        line["workloads"] = extra
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(strip_args(sys.argv[1:]), wl)
    return line


# ---------------------------------------------------------------------------- reference arm

def instrumented_stage_ms(layer, L_d, x_d, r_d, stages, steps):
    """Mean device time of every stage over one replay of a graph of `steps`
    layer steps with timing nodes around each stage (not the timed region)."""
    import torch
    mk = lambda: (torch.cuda.Event(enable_timing=True, external=True),  # noqa: E731
                  torch.cuda.Event(enable_timing=True, external=True))
    ev = [{s: mk() for s in stages} for _ in range(steps)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(steps):
            layer.forward_stages(L_d, x_d, r_d, events=ev[i])
    graph.replay()  # uploads the graph
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    return {s: statistics.mean(e[s][0].elapsed_time(e[s][1]) for e in ev) for s in stages}


def stage_alone_ms(layer, L_d, x_d, r_d, stages, reps):
    """Per-launch device time of every stage run alone: a graph of `reps`
    back-to-back launches of that stage on the layer's own buffers (no other
    stage, no timing node between the launches), replayed once to upload it
    and once under CUDA events.  The in-step figures carry the cost of the
    timing nodes around each stage; these do not."""
    import torch
    st = torch.cuda.current_stream()
    out = {}
    for name in stages:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(reps):
                layer.run_stage(name, L_d, x_d, r_d, layer.out, torch.cuda.current_stream())
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        graph.replay()
        e1.record(st)
        torch.cuda.synchronize()
        out[name] = e0.elapsed_time(e1) / reps
        del graph
    return out


def run_reference(args):
    """The oracle as it stands, timed on every host core: K steps after W
    warm-up steps, each a bounded sample of the workload (oracle_worker)."""
    world, rank, _ = dist_info()
    if rank != 0:
        return None
    wl = workload(args)
    argv = strip_args(sys.argv[1:])
    ncpu = os.cpu_count() or 1
    experts = 2
    r = run_oracle(argv, ncpu, steps=args.steps + args.warmup, experts_per_step=experts)
    timed = r["steps"][args.warmup:]
    tokens = sum(s["tokens"] for s in timed)
    secs = sum(s["seconds"] for s in timed)
    value = tokens / secs if secs > 0 else 0.0
    sample = (oracle_sample_text(wl, experts, len(timed), r["n_sub"]) +
              f"; {ncpu} threads in the BLAS calls")
    return {
        "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / len(timed) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": workload_config(wl),
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": ncpu,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    if args.oracle_worker:
        print(json.dumps(oracle_worker(json.loads(args.oracle_worker))))
        return
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
