"""Host-side logic of bench.py (CPU only): the multi-rank reduction over gloo
with two ranks, the whole-job rate, and the reference arm's non-zero ranks."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r timed (1 + r, 10 - r, 5) ms: the job takes the slowest of each
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 5.0], torch.device("cpu"), world)
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        assert out[r] == [2.0, 10.0, 5.0]


def test_single_rank_and_job_rate():
    assert bench.max_over_ranks([3, 4.5], None, 1) == [3.0, 4.5]
    # two replicas of 2048 tokens each in 0.5 ms (the slowest): 8.192 M tokens/s
    assert bench.job_rate(2048, 2, 0.5) == pytest.approx(8.192e6)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "1"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_json_line_on_rank_zero():
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_fp32", "--steps", "1", "--warmup", "1"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    import json
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["config"]["workload"] == "tiny_fp32" and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


@pytest.mark.parametrize("opts,router,name", [
    (["--straight-through"], {"gumbel_straight_through": True}, "tiny_fp32+gumbelST"),
    (["--padding-mask", "--temperature", "0.5"], {"padding_mask": True, "temperature": 0.5},
     "tiny_fp32+tau0.5+mask"),
    (["--raw-gates", "--top-k", "1"], {"normalize_gates": False}, "tiny_fp32+k1+rawgates"),
])
def test_reference_arm_router_variants(opts, router, name):
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_fp32", "--steps", "1", "--warmup", "1", *opts],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    import json
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["config"]["workload"] == name and d["value"] > 0
    for k, v in router.items():
        assert d["config"]["router"][k] == v, k


def test_roofline_traffic_comes_from_the_matching_profile(tmp_path, monkeypatch):
    """`roofline.traffic` is read from the committed per-workload ncu summary only when
    it names the same workload and the grouped-GEMM sources still hash to its digest."""
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    dig = bench.gemm_source_digest()
    p = tmp_path / "tc_grouped_gemm_mixtral_bf16.md"
    p.write_text(f"workload: mixtral_bf16\ntraffic_bytes_per_step: 175535728896\n"
                 f"gemm_source_sha256: {dig}\n")
    assert bench.gemm_traffic_from_profile("mixtral_bf16") == 175535728896.0
    # another workload's profile, a stale digest, or no profile: no traffic figure
    assert bench.gemm_traffic_from_profile("llama4_bf16") is None
    p.write_text("workload: mixtral_bf16\ntraffic_bytes_per_step: 1\ngemm_source_sha256: " + "0" * 64 + "\n")
    assert bench.gemm_traffic_from_profile("mixtral_bf16") is None
    p.write_text(f"workload: llama4_bf16\ntraffic_bytes_per_step: 1\ngemm_source_sha256: {dig}\n")
    assert bench.gemm_traffic_from_profile("mixtral_bf16") is None


def test_committed_gemm_profiles_name_their_workload():
    """Every committed GEMM traffic summary is parseable and keyed by its own workload."""
    import re
    for name in os.listdir(bench.PROFILES):
        m = re.fullmatch(r"tc_grouped_gemm_(\w+)\.md", name)
        if not m:
            continue
        txt = open(os.path.join(bench.PROFILES, name)).read()
        if "traffic_bytes_per_step:" not in txt:
            continue
        wl = re.search(r"workload:\s*(\S+)", txt).group(1)
        assert bench.gemm_profile_path(wl).endswith(name)
        assert re.search(r"gemm_source_sha256:\s*[0-9a-f]{64}", txt)
