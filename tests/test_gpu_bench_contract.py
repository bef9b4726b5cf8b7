"""bench.py on the GPU: one short run on the GPT-2-small workload prints one
JSON line with the benchmark contract's keys, and the figures hang together
(params/s from the step time, the roofline from its parts, this library's
kernels launched in the timed region, the end-to-end copy bytes counted from
the gradients)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_keeps_the_contract(zero_lib):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "gpt2small_n4",
                        "--steps", "5", "--warmup", "3", "--no-cpu-baseline", "--e2e-steps", "2",
                        "--sequence"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
                "cpu_baseline", "e2e", "gpu_launches", "clocks", "sequence"):
        assert key in d, key
    assert d["unit"] == "params/s" and d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    cfg = d["config"]
    assert cfg["workload"] == "gpt2small_n4" and cfg["N"] == 4
    # params/s is the parameter count over the step time
    assert abs(d["value"] - cfg["psi"] / (d["ms_per_step"] / 1e3)) <= 1e-3 * d["value"]
    rf = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic", "frac_of_nominal"):
        assert key in rf, key
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert 0.3 < rf["frac"] < 1.3
    assert d["gpu_launches"] >= d["steps"] * rf["launches_per_step"]
    e2e = d["e2e"]
    if "unavailable" not in e2e:
        # every rank's BF16 gradient for the padded vector, copied each step
        assert e2e["h2d_bytes_per_step"] == cfg["N"] * cfg["psi_pad"] * 2
        assert e2e["d2h_bytes_per_step"] == 16 and e2e["value"] > 0
    seq = d["sequence"]
    assert seq["steps"] == 10 and len(seq["ms"]) == 10 and seq["skipped_steps"] == []
    c = d["clocks"]
    assert "sm_mhz" in c and "reasons" in c


def test_profile_graph_replays_one_real_step(zero_lib):
    """--profile-graph captures one step as a CUDA graph and replays it between
    cudaProfilerStart/Stop (the range ncu measures as a unit); the replayed step
    applies, and the timed steps after it still run and keep the line's shape."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "gpt2small_n4",
                        "--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--no-e2e",
                        "--no-sequence", "--policy", "device", "--profile-graph"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    assert "graph step:" in r.stderr
    ms = float(r.stderr.split("graph step:")[1].split("ms")[0])
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    d = json.loads(lines[-1])
    # the replayed step does the work of an eager one, within launch overheads
    assert 0.5 * d["ms_per_step"] < ms < 3.0 * d["ms_per_step"], (ms, d["ms_per_step"])
    assert d["config"]["step_policy"] == "device"
