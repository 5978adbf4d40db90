"""bench.py keeps its output contract: one JSON line with the metric, the
whole-job value, the timing record, the roofline of the dominant kernel, the
end-to-end figure through the host-buffer API, the kernel-launch count and
the SM clocks sampled during the timed region."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bench_line(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                         capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("extra", [[], ["--eager"], ["--workload", "correlated_placed",
                                                      "--tokens", "2048"],
                                   ["--others", "tiny"]])
def test_bench_json_contract(extra):
    args = ["--workload", "tiny", "--steps", "3", "--warmup", "3", "--no-cpu-baseline",
            "--e2e-steps", "3"]
    d = bench_line(*(args + extra))
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks", "stages"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["dtype"] == "bf16"
    assert "workload" in d["config"]
    roof = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in roof, key
    assert roof["bound"] in ("hbm", "tensor") and roof["frac"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 2e-3
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    if "--others" in extra:
        # one compact entry per extra workload, measured like the headline
        o = d["workloads"]["tiny"]
        for key in ("value", "unit", "ms_per_step", "config", "roofline", "stages",
                    "dispatch_rows", "gpu_launches", "clocks"):
            assert key in o, key
        assert o["value"] > 0 and o["roofline"]["frac"] > 0
    # every stage is also timed alone (graph mode only)
    if "--eager" not in extra:
        for name, st in d["stages"].items():
            assert st["alone_ms"] > 0 and st["alone_hbm_frac"] >= 0, name
    rows = d["dispatch_rows"]
    for key in ("plain", "dedup", "dedup_reduction", "ranks_per_token", "same_rank_share",
                "max_over_mean_expert_load"):
        assert key in rows, key
    assert abs(rows["ranks_per_token"] - rows["dedup"] / d["config"]["N"]) < 1e-3
