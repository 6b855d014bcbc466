"""The benchmark's JSON line on the GPU: one short run of the small workload through
bench.py, checked for the fields and the internal consistency its consumers rely on
(time-like figures inside the step, the roofline against the measured peaks, launches
counted from the captured step, copies counted from the tensors moved)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_line_of_the_small_workload():
    j = _run("--workload", "small_bf16", "--steps", "5", "--warmup", "3", "--no-cpu-baseline")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "clocks", "gpu_launches", "stages_ms", "hbm_gbs", "routing"):
        assert key in j, key
    assert j["n_gpus"] == 1 and j["steps"] == 5 and j["warmup"] >= 3
    assert j["config"]["workload"] == "small_bf16" and j["config"]["T"] == 2048
    # throughput is the batch over the step time
    assert j["value"] == pytest.approx(2048 / (j["ms_per_step"] * 1e-3), rel=1e-6)
    r = j["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-9)
    assert 0 < r["gemm_ms_per_step"] <= j["ms_per_step"]          # measured inside the step
    assert 0 < r["frac"] < 1.5
    # the small workload's profile names it, so its traffic is reported for unchanged sources
    assert r["traffic"] is None or r["traffic"] > 0
    # launches: the captured step's count, times the timed steps
    assert j["gpu_launches"] == 5 * j["launches_per_step"] and j["launches_per_step"] >= 10
    # end to end: x and dout in, out and dx back, bf16
    e = j["e2e"]
    assert e["h2d_bytes_per_step"] == 2 * 2048 * 1024 * 2
    assert e["d2h_bytes_per_step"] == 2 * 2048 * 1024 * 2
    assert 0 < e["value"] < j["value"]                            # copies cost time
    assert set(j["stages_ms"]) == {"route", "permute", "grouped_ffn", "combine", "combine_bwd",
                                   "grouped_ffn_bwd", "router_bwd"}
    ro = j["routing"]
    assert ro["kept_assignments"] + ro["dropped_assignments"] == 2048 * 2
    assert j["clocks"]["sm_max_mhz"] > 0
