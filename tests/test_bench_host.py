"""Host-side logic of bench.py: argument handling, algorithmic byte counts and
the multi-rank timing reduction (world_size 2 over gloo on the CPU)."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    got = bench.max_over_ranks(10.0 + rank, world)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_world2_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 11.0, 1: 11.0}


def test_strip_args_keeps_the_workload():
    argv = ["--impl", "reference", "--workload", "mixtral", "--steps", "5", "--tokens", "64",
            "--no-cpu-baseline"]
    assert bench.strip_args(argv) == ["--workload", "mixtral", "--tokens", "64"]


def test_algorithmic_bytes_of_the_deepseek_layer():
    args = bench.parse_args([])
    wl = bench.workload(args)
    alg = bench.algorithmic(wl, R_d=0)
    # gate/up streams 2 * E * I * H bf16 weights plus its rows in and out
    assert alg["gate_up"]["bytes"] == 2 * 256 * 2048 * 7168 * 2 + 32768 * 7168 * 2 + 32768 * 2048 * 2
    assert alg["gate_up"]["flops"] == 4 * 32768 * 7168 * 2048
    assert alg["dispatch"]["bytes"] == 4096 * 7168 * 2 * (1 + 8)
    # with the dispatch fused into it, gate/up reads each token row of x once
    fused = bench.algorithmic(wl, R_d=0, fused_dispatch=True)
    assert fused["gate_up"]["bytes"] == (2 * 256 * 2048 * 7168 * 2 + 4096 * 7168 * 2 +
                                         32768 * 2048 * 2)


def test_algorithmic_bytes_of_the_fused_ffn_and_its_roofline_stage():
    """The fused expert FFN's algorithmic bytes: all three weight matrices, the
    rows it gathers once (x when plain, the dedup rows when dedup) and y out;
    h, which never leaves the SM, is not counted.  Where the layer fuses the
    FFN, the roofline object describes that kernel."""
    import types
    wl = bench.workload(bench.parse_args(["--workload", "tiny"]))
    E, H, I, N, k = wl.E, wl.H, wl.I, wl.N, wl.k
    alg = bench.algorithmic(wl, R_d=0, fused_dispatch=True)
    assert alg["ffn"]["bytes"] == 3 * E * I * H * 2 + N * H * 2 + N * k * H * 2
    assert alg["ffn"]["flops"] == alg["gate_up"]["flops"] + alg["down"]["flops"]
    assert bench.dominant_stage(types.SimpleNamespace(fused_ffn=True)) == "ffn"
    assert bench.dominant_stage(types.SimpleNamespace(fused_ffn=False)) == "gate_up"


def test_workload_overrides():
    wl = bench.workload(bench.parse_args(["--tokens", "512", "--experts", "32"]))
    assert (wl.N, wl.E, wl.W, wl.H) == (512, 32, 8, 7168)


def test_recorded_traffic_follows_the_gemm_sources(tmp_path, monkeypatch):
    """roofline.traffic is reported only while the GEMM sources keep the bytes
    the capture was taken on, and only for the captured workload."""
    import json
    import shutil
    for rel in bench.TRAFFIC_SOURCES:
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, rel), dst)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"sources_sha256_prefix": bench.sources_digest(),
           "gate_up": {"mixtral": {"dram_bytes": 123}}}
    (tmp_path / "profiles" / "gemm_traffic.json").write_text(json.dumps(rec))
    args = bench.parse_args(["--workload", "mixtral"])
    assert bench.recorded_traffic(bench.workload(args)) == 123
    assert bench.recorded_traffic(bench.workload(bench.parse_args([]))) is None
    # a comment does not change the code the capture was taken on; code does
    with open(tmp_path / bench.TRAFFIC_SOURCES[2], "a") as f:
        f.write("// a comment\n")
    assert bench.recorded_traffic(bench.workload(args)) == 123
    with open(tmp_path / bench.TRAFFIC_SOURCES[2], "a") as f:
        f.write("static int changed_code;\n")
    assert bench.recorded_traffic(bench.workload(args)) is None


def test_oracle_worker_times_every_stage_of_a_step():
    """The CPU baseline's worker times route, layout, dispatch, the sampled
    expert FFN (scaled to all rows) and the combine, in a one-thread process."""
    r = bench.run_oracle(["--workload", "tiny"], threads=1, steps=2, experts_per_step=2)
    assert r["threads"] == 1 and len(r["steps"]) == 2
    for st in r["steps"]:
        assert set(st["stage_s"]) == {"route", "layout", "dispatch", "ffn", "combine"}
        assert st["tokens"] == 64 and st["seconds"] > 0
        assert st["rows_sampled"] > 0 and len(st["experts"]) == 2
    # successive steps sample different experts of one permutation
    assert r["steps"][0]["experts"] != r["steps"][1]["experts"]


def test_oracle_worker_dedup_combine_sample():
    r = bench.run_oracle(["--workload", "correlated_placed", "--tokens", "300"], threads=1,
                         steps=1, experts_per_step=1)
    assert r["steps"][0]["tokens"] == 300 and r["n_sub"] == 300


def test_reference_arm_prints_its_contract_line():
    """bench.py --impl reference: the oracle timed on the host cores, one JSON
    line with the same metric and workload keys as the repo's arm, marked as
    the reference, with its cpu_baseline and zero-copy e2e."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, cwd=root, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [line for line in out.stdout.splitlines() if line.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["steps"] == 2 and d["warmup"] == 1 and d["value"] > 0
    assert d["config"]["workload"] == "tiny" and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
