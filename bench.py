"""Benchmark of the sparse MoE layer (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = the whole hot path on one batch of synthetic tokens: router,
permutation, grouped expert FFN, combine (forward) and the full backward
(combine-bwd, grouped FFN backward, router backward), all through the C ABI,
replayed as one CUDA graph (the ABI does no host sync and no allocation, so
the step is capturable).  The default workload is the Mixtral-shaped layer at
T = 65536 tokens (d 4096, f 14336, E 8, top-2, SwiGLU), the largest shape.

Timing: the step graph carries external CUDA events around its two grouped-GEMM
calls, so the grouped-GEMM time of the roofline is measured inside the very
replays whose duration gives ms_per_step (it cannot exceed the step).  Inputs
and weights are resident in HBM before the timed region; L2 is flushed before
every timed step, outside its event pair (a 512 MB write, then a 1 GB read that
also pushes the written lines back to DRAM before the step starts).  Per-stage times
come from a second capture of the step with an event between every two C-ABI calls,
replayed after the same flush (reported beside the line, not used for the roofline).
Under torchrun each rank runs an independent replica on its own GPU (the
layer has no exchange step on one GPU); rank 0 prints one JSON line with the
whole-job tokens/s (max step time over ranks).

`e2e` is the same step through the public layer API with pinned host buffers,
every transfer inside the timed region: x copied in, the forward, dout copied
in on a copy stream during the forward, out copied back during the backward,
dx copied back at the end.

--impl reference times the fp64 CPU oracle (the layer's plain definition) on
the host cores, on a bounded token sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time
from dataclasses import replace

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import moe_inputs  # noqa: E402

METRIC = "MoE layer tokens/sec fwd and fwd+bwd on 1 GB300; grouped-GEMM % of bf16 peak"
DEFAULT_WORKLOAD = "mixtral_bf16"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILES = os.path.join(ROOT, "profiles")
GEMM_SOURCES = [os.path.join(ROOT, "top_routing_expert_moe_gb300", "csrc", f)
                for f in ("gemm_tc.cu", "tma.cuh", "common.cuh")]
SUSTAINED_AFTER_S = 1.0   # timed regions at least this long run under the power cap
GEMM_LAUNCHES_PER_STEP = 4  # GEMM1, GEMM2, {dgrad2 || dW_down}, {dW_up [|| dW_gate] || dgrad1}


# ----------------------------------------------------------------------------- helpers
def max_over_ranks(values, device, world):
    """Per-rank timings -> their maximum over all ranks (the job ends with the
    slowest replica); identity on one rank."""
    if world == 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_rate(units_per_rank, world, ms):
    """Whole-job rate: every rank processed units_per_rank in (at most) ms."""
    return units_per_rank * world / (ms * 1e-3)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def pick_bf16_peak(peaks, timed_region_s):
    """The burst figure for a short timed region, the sustained (power-capped)
    one once the timed region lasts SUSTAINED_AFTER_S or more."""
    if timed_region_s >= SUSTAINED_AFTER_S and "bf16_tflops_sustained" in peaks:
        return float(peaks["bf16_tflops_sustained"]), "sustained"
    return float(peaks["bf16_tflops"]), "burst"


def algorithmic_work(w, A_kept: int):
    """FLOPs of the grouped GEMMs and bytes of the HBM-bound kernels per step."""
    s = 2 if w.dtype == "bf16" else 4
    T, d, f, E, k = w.T, w.d, w.f, w.E, w.k
    A = T * k
    # routed experts on the kept assignments, plus the shared experts on every token
    fwd = (6 if w.swiglu else 4) * (A_kept * d * f + T * d * w.f_shared)
    return dict(
        gemm_fwd_flop=fwd, gemm_bwd_flop=2 * fwd,
        route_bytes=T * d * s + d * E * s + T * (4 * E + 8 * k),
        permute_bytes=2 * A_kept * d * s + 8 * A,
        combine_bytes=A_kept * d * s + T * d * s + 8 * A + (T * d * s if w.f_shared else 0))


def gemm_source_digest() -> str:
    h = hashlib.sha256()
    for p in GEMM_SOURCES:
        with open(p, "rb") as fh:
            h.update(os.path.basename(p).encode() + fh.read())
    return h.hexdigest()


def gemm_profile_path(workload: str) -> str:
    return os.path.join(PROFILES, "tc_grouped_gemm_" + re.sub(r"[^A-Za-z0-9_]", "_", workload) + ".md")


def gemm_traffic_from_profile(workload: str):
    """DRAM bytes of all grouped-GEMM launches of one step of this workload (the unit
    of `achieved`) from its committed ncu summary; None when there is none or the
    kernel source changed since."""
    path = gemm_profile_path(workload)
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"traffic_bytes_per_step:\s*([0-9.eE+]+)", txt)
    h = re.search(r"gemm_source_sha256:\s*([0-9a-f]{64})", txt)
    wl = re.search(r"workload:\s*(\S+)", txt)
    if not m or not h or not wl or wl.group(1) != workload:
        return None
    return float(m.group(1)) if gemm_source_digest() == h.group(1) else None


class ClockSampler:
    """nvidia-smi sampling around the timed region (SM clock, throttle reasons)."""
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        # raw samples: a temporary file unless MOE_BENCH_CLOCKS_DIR names a folder to keep them in
        out_dir = os.environ.get("MOE_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"moe_bench_clocks_{os.getpid()}.csv")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as fh:
            lines = fh.readlines()
        if not os.environ.get("MOE_BENCH_CLOCKS_DIR"):
            try:
                os.remove(self.path)
            except OSError:
                pass
        rows = []
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, float(parts[1]), float(parts[2]), parts[4:]))
            except Exception:
                continue
        if not rows:
            return None
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        window = "timed_region"
        if not inside:
            inside = sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:3]
            window = "nearest_samples"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[3][1:]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


class StepEvent:
    """A timing event that may also be recorded while a stream is captured: it
    becomes an external event node of the graph, so every replay re-records it
    and the graph times its own parts.  torch's external events where torch
    offers them, else the driver's cuEventRecordWithFlags(..., EXTERNAL)."""
    _drv = None

    def __init__(self):
        import torch
        self.ev = None
        try:
            self.ev = torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            drv = StepEvent._driver()
            self.h = ctypes.c_void_p()
            if drv.cuEventCreate(ctypes.byref(self.h), 0) != 0:
                raise RuntimeError("cuEventCreate failed")

    @staticmethod
    def _driver():
        if StepEvent._drv is None:
            StepEvent._drv = ctypes.CDLL("libcuda.so.1")
        return StepEvent._drv

    def record(self, stream):
        if self.ev is not None:
            self.ev.record(stream)
        elif StepEvent._driver().cuEventRecordWithFlags(self.h, ctypes.c_void_p(stream.cuda_stream),
                                                        1) != 0:
            raise RuntimeError("cuEventRecordWithFlags failed")

    def elapsed_ms(self, later: "StepEvent") -> float:
        if self.ev is not None:
            return float(self.ev.elapsed_time(later.ev))
        ms = ctypes.c_float()
        drv = StepEvent._driver()
        fn = getattr(drv, "cuEventElapsedTime_v2", None) or drv.cuEventElapsedTime
        if fn(ctypes.byref(ms), self.h, later.h) != 0:
            raise RuntimeError("cuEventElapsedTime failed")
        return float(ms.value)


# ----------------------------------------------------------------------------- oracle leg
def router_variant(args=None) -> dict:
    """The router options of a run (softmax temperature, raw or renormalised gates, a
    padding mask, Gumbel top-k with the straight-through estimator)."""
    if args is None:
        return dict(temperature=1.0, normalize=True, mask=False, straight_through=False)
    return dict(temperature=args.temperature, normalize=not args.raw_gates,
                mask=args.padding_mask, straight_through=args.straight_through)


def variant_inputs(w, v: dict, seed: int):
    """Seeded selection noise (Gumbel draws) and token mask of a router variant."""
    gum = moe_inputs.gumbel(seed, w.T, w.E) if v["straight_through"] else None
    mask = moe_inputs.padding_mask(seed, w.T) if v["mask"] else None
    return gum, mask


class OracleInputs:
    """A workload's seeded inputs for the oracle: the weights converted to fp64
    once; samples take the first T_s tokens of x, dout and the noise (the GPU
    arm's own draws when ``inp`` is given, else drawn from the same seed)."""

    def __init__(self, w, v: dict, seed: int = 0, inp=None, max_tokens=None):
        import oracle
        self.oracle, self.w, self.v = oracle, w, v
        self.cap = min(w.T, max_tokens or w.T)
        if inp is None:
            inp = moe_inputs.make_inputs(replace(w, T=self.cap), seed)
        self.tok = {k_: inp.get(k_) for k_ in ("x", "dout", "noise")}
        self.weights = {k_: moe_inputs.as_f64(a, w.dtype if k_ != "bias" else "fp32")
                        for k_, a in inp.items() if k_ not in self.tok}
        gum, mask = variant_inputs(w, v, seed) if (v["straight_through"] or v["mask"]) else (None, None)
        self.gum, self.mask = gum, mask

    def sample(self, T_s: int) -> "OracleSample":
        return OracleSample(self, int(min(T_s, self.cap)))


class OracleSample:
    """The first T_s tokens of an OracleInputs, ready to run forward + backward."""

    def __init__(self, src: OracleInputs, T_s: int):
        w, v, o_ = src.w, src.v, src.oracle
        self.oracle, self.T_s = o_, T_s
        f = dict(src.weights)
        for k_, a in src.tok.items():
            f[k_] = None if a is None else moe_inputs.as_f64(a[:T_s], w.dtype if k_ != "noise" else "fp32")
        self.f64 = f
        self.noise = moe_inputs.as_f64(src.gum[:T_s], "fp32") if src.gum is not None else f["noise"]
        self.mask = src.mask[:T_s] if src.mask is not None else None
        self.cfg = o_.OracleConfig(T=T_s, d=w.d, f=w.f, E=w.E, k=w.k,
                                   capacity_factor=float(np.float32(w.capacity_factor)),
                                   swiglu=w.swiglu, aux_coef=w.aux_coef, pad_m=128,
                                   f_shared=w.f_shared, normalize_gates=v["normalize"],
                                   temperature=float(np.float32(v["temperature"])),
                                   straight_through=v["straight_through"])

    def run(self) -> float:
        """One oracle forward + backward; its wall time in seconds."""
        o_, f = self.oracle, self.f64
        sh = dict(Wup_s=f.get("W_up_s"), Wdown_s=f.get("W_down_s"), Wgate_s=f.get("W_gate_s"))
        t0 = time.perf_counter()
        o = o_.forward(self.cfg, f["x"], f["W_r"], f["W_up"], f["W_down"], Wgate=f["W_gate"],
                       bias=f["bias"], noise=self.noise, mask=self.mask, **sh)
        o_.backward(self.cfg, f["x"], f["W_r"], f["W_up"], f["W_down"], o["logits"],
                    o["topk_idx"], o["gate"], o["slot_of"], f["dout"], Wgate=f["W_gate"],
                    with_bias=f["bias"] is not None, **sh)
        return time.perf_counter() - t0


def oracle_sample_tokens(src: OracleInputs, budget_s: float) -> int:
    """Token count whose oracle fwd+bwd takes about budget_s on this host: two
    pilot runs give the fixed cost (the weight gradients are written whatever
    the token count) and the cost per token."""
    cap = src.cap
    n1, n2 = min(8, cap), min(32, cap)
    s1 = src.sample(n1)
    t1 = min(s1.run(), s1.run())
    if n2 == n1:
        return n1
    t2 = src.sample(n2).run()
    per_tok = max((t2 - t1) / (n2 - n1), 1e-6)
    fixed = max(t1 - per_tok * n1, 0.0)
    return int(max(n1, min(cap, (budget_s - fixed) / per_tok)))


def oracle_cores():
    import oracle
    return oracle.max_threads()


def cpu_model() -> str:
    """The host CPU's model name as the kernel reports it (lscpu's source), or the
    architecture when the name is not listed (some Arm kernels omit it)."""
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


def workload_config(w, v: dict | None = None):
    v = v or router_variant()
    return {"workload": w.name, "T": w.T, "d_model": w.d, "d_ff": w.f, "experts": w.E,
            "top_k": w.k, "capacity_factor": w.capacity_factor,
            "ffn": "swiglu" if w.swiglu else "silu", "gate_noise_std": w.noise_std,
            "zipf_router_bias": w.zipf_bias, "aux_coef": w.aux_coef, "f_shared": w.f_shared,
            "router": {"temperature": v["temperature"], "normalize_gates": v["normalize"],
                       "padding_mask": v["mask"], "gumbel_straight_through": v["straight_through"]},
            "l2": "GPU arm: flushed before every step (512 MB write, then 1 GB read)",
            "parallelism": "replicas (one independent layer per GPU)"}


def run_reference(args, w):
    ws_, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    v = router_variant(args)
    # the sample's inputs: the first tokens of the same seeded draws the GPU arm uses
    src = OracleInputs(w, v, args.seed, max_tokens=4096)
    T_s = oracle_sample_tokens(src, args.ref_budget_s)
    samp = src.sample(T_s)
    for _ in range(args.warmup):
        samp.run()
    times = [samp.run() for _ in range(args.steps)]
    step_s = statistics.mean(times)
    tok_s = T_s / step_s
    sample = (f"oracle fp64 fwd+bwd on the first {T_s} tokens of {w.name} (same d, f, E, k, "
              f"capacity factor, weights and seed), per step")
    line = {"impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * step_s, "tokens_per_step": T_s,
            "ms_per_full_batch_extrapolated": 1e3 * step_s * w.T / T_s,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded normals, random-init weights)",
            "config": workload_config(w, v),
            "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": oracle_cores(),
                             "cpu_model": cpu_model(), "kind": "oracle", "sample": sample},
            "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def cpu_baseline_leg(w, v, inp, seed, budget_s, one_core_budget_s):
    """The oracle as it stands on a bounded sample of the workload: on every host
    core, then on one core."""
    import oracle
    oracle.build()
    cores = oracle_cores()
    src = OracleInputs(w, v, seed, inp=inp)
    T_s = oracle_sample_tokens(src, budget_s)
    t_all = src.sample(T_s).run()
    out = {"value": T_s / t_all, "unit": "tokens/s", "cores": cores, "cpu_model": cpu_model(),
           "kind": "oracle",
           "sample": f"oracle fp64 fwd+bwd on the first {T_s} tokens of {w.name} "
                     f"(same d, f, E, k, weights), {t_all:.1f} s"}
    if one_core_budget_s > 0:
        oracle.set_threads(1)
        try:
            T_1 = oracle_sample_tokens(src, one_core_budget_s)
            t_1 = src.sample(T_1).run()
        finally:
            oracle.set_threads(cores)
        out["one_core"] = {"value": T_1 / t_1, "unit": "tokens/s", "cores": 1,
                           "sample": f"first {T_1} tokens, {t_1:.1f} s"}
    return out


# ----------------------------------------------------------------------------- GPU leg
def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import top_routing_expert_moe_gb300 as moe

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    moe.load_library()

    v = router_variant(args)
    cfg = moe.config_for(w, normalize=v["normalize"], temperature=v["temperature"],
                         straight_through=v["straight_through"])
    inp = moe_inputs.make_inputs(w, args.seed + rank)
    gum, mask_np = variant_inputs(w, v, args.seed + rank)
    dt = w.dtype
    td = moe.tensor_from_numpy
    x = td(inp["x"], dt, dev)
    Wr = td(inp["W_r"], dt, dev)
    Wu = td(inp["W_up"], dt, dev)
    Wg = td(inp["W_gate"], dt, dev)
    Wd = td(inp["W_down"], dt, dev)
    b = td(inp["bias"], "fp32", dev)
    nz = td(gum if gum is not None else inp["noise"], "fp32", dev)
    mk = torch.from_numpy(mask_np).to(dev) if mask_np is not None else None
    dout = td(inp["dout"], dt, dev)
    L = moe.MoELayer(cfg, device=dev)
    g = L.grads()
    shared_w = None
    sh_f = sh_b = None
    if w.f_shared > 0:             # the shared experts' FFN (same launches as the routed one)
        shared_w = (td(inp["W_up_s"], dt, dev), td(inp["W_down_s"], dt, dev),
                    td(inp.get("W_gate_s"), dt, dev))
        Ts = L.shared_rows
        sh_f = moe.shared_block(x=x, W_up=shared_w[0], W_down=shared_w[1], W_gate=shared_w[2],
                                h=L.h_shared, act=L.act_shared, y=L.y_shared)
        sh_b = moe.shared_block(
            x=x, W_up=shared_w[0], W_down=shared_w[1], W_gate=shared_w[2], h=L.h_shared,
            act=L.act_shared, y=L.y_shared, dout=dout,
            dh=torch.empty(cfg.nh, Ts, w.f_shared, dtype=cfg.torch_dtype, device=dev),
            dx=torch.empty(Ts, w.d, dtype=cfg.torch_dtype, device=dev),
            dW_up=g["dW_up_s"], dW_gate=g["dW_gate_s"], dW_down=g["dW_down_s"])
    st = torch.cuda.Stream(dev)           # a side stream: graphs cannot capture the default one
    flush_w = torch.empty(512 * 2**20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(256 * 2**20, dtype=torch.int32, device=dev)

    def flush_l2():
        """Evict L2 before a timed step: write 512 MB, then read 1 GB of another
        buffer so the written lines are also written back to DRAM here, outside
        the step's events (otherwise the first timed kernel pays for them)."""
        flush_w.zero_()
        flush_r.sum()
    R = L.rows_cap
    bw = dict(dy=torch.empty(R, w.d, dtype=cfg.torch_dtype, device=dev),
              dgate=torch.empty(w.T, w.k, dtype=torch.float32, device=dev),
              dh=torch.empty(cfg.nh, R, w.f, dtype=cfg.torch_dtype, device=dev),
              dxp=torch.empty(R, w.d, dtype=cfg.torch_dtype, device=dev),
              dlogits=torch.empty(w.T, w.E, dtype=torch.float32, device=dev))
    torch.cuda.synchronize(dev)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def rec(evs, i):
        if evs is not None:
            evs[i].record(st)

    # one step through the C ABI; optional events around each call (all on `st`);
    # gev: four step events around the two grouped-GEMM calls
    def forward(evs=None, gev=None):
        rec(evs, 0)
        moe.moe_route(cfg, x, Wr, b, nz, mk, L.logits, L.topk_idx, L.gate, L.counts, L.stats, L.ws, st)
        rec(evs, 1)
        moe.moe_permute(cfg, x, L.topk_idx, L.x_perm, L.perm_token, L.slot_of, L.kept, L.offsets,
                        L.stats, L.ws, st)
        rec(evs, 2)
        if gev:
            gev[0].record(st)
        moe.moe_grouped_ffn(cfg, L.x_perm, L.offsets, Wu, Wg, Wd, L.h_saved, L.act, L.y_perm,
                            L.ws, st, shared=sh_f)
        if gev:
            gev[1].record(st)
        rec(evs, 3)
        moe.moe_combine(cfg, L.y_perm, L.slot_of, L.gate, L.out, st, shared=sh_f)
        rec(evs, 4)

    def backward(evs=None, gev=None):
        moe.moe_combine_backward(cfg, dout, L.y_perm, L.gate, L.slot_of, L.perm_token, L.offsets,
                                 bw["dy"], bw["dgate"], st)
        rec(evs, 5)
        if gev:
            gev[2].record(st)
        moe.moe_grouped_ffn_backward(cfg, L.x_perm, L.offsets, Wu, Wg, Wd, L.h_saved, L.act,
                                     bw["dy"], bw["dh"], bw["dxp"], g["dW_up"], g["dW_gate"],
                                     g["dW_down"], L.ws, st, shared=sh_b)
        if gev:
            gev[3].record(st)
        rec(evs, 6)
        moe.moe_router_backward(cfg, x, Wr, L.logits, L.topk_idx, L.gate, L.slot_of, bw["dgate"],
                                bw["dxp"], L.stats, g["dx"], g["dW_r"],
                                g["dbias"] if b is not None else None, bw["dlogits"], L.ws, st,
                                shared=sh_b)
        rec(evs, 7)

    def step(evs=None, gev=None):
        forward(evs, gev)
        backward(evs, gev)

    with torch.cuda.stream(st):
        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize(dev)
        status = moe.last_device_status(st)
        if status != 0:
            raise RuntimeError(f"device status after warm-up: {moe.error_string(status)}")
        A_kept = int(L.kept.sum().item())
        stats = L.stats.cpu().tolist()
        work = algorithmic_work(w, A_kept)

        # the step (with its grouped-GEMM events) and the forward as CUDA graphs (the C ABI
        # is capturable: no host sync, no allocation); their kernel count per replay is the
        # capture's launch count
        gev = [StepEvent() for _ in range(4)]
        graph, fgraph = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        n0 = moe.launch_count()
        with torch.cuda.graph(graph, stream=st):
            step(gev=gev)
        launches_per_step = moe.launch_count() - n0
        with torch.cuda.graph(fgraph, stream=st):
            forward()
        torch.cuda.synchronize(dev)
        for _ in range(3):
            graph.replay()
            fgraph.replay()
        torch.cuda.synchronize(dev)

        sampler = ClockSampler(local)
        time.sleep(0.3)
        step_evs = [(ev(), ev()) for _ in range(args.steps)]
        gemm_ms_steps = []
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t_wall0 = time.time()
        for i in range(args.steps):
            flush_l2()                      # outside the step's events
            step_evs[i][0].record(st)
            graph.replay()
            step_evs[i][1].record(st)
            st.synchronize()                # the next replay re-records the step's GEMM events
            gemm_ms_steps.append(gev[0].elapsed_ms(gev[1]) + gev[2].elapsed_ms(gev[3]))
        torch.cuda.synchronize(dev)
        t_wall1 = time.time()
        if world > 1:
            dist.barrier()
        clocks = sampler.stop(t_wall0, t_wall1)
        step_ms = [a.elapsed_time(c) for a, c in step_evs]
        ms_local = float(np.mean(step_ms))
        gemm_ms_local = float(np.mean(gemm_ms_steps))
        assert all(gm <= sm for gm, sm in zip(gemm_ms_steps, step_ms)), "GEMM events outside the step"
        status = moe.last_device_status(st)
        if status != 0:
            raise RuntimeError(f"device status after the timed steps: {moe.error_string(status)}")

        # forward only (graph)
        fwd_evs = [(ev(), ev()) for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2()
            fwd_evs[i][0].record(st)
            fgraph.replay()
            fwd_evs[i][1].record(st)
        torch.cuda.synchronize(dev)
        fwd_ms = float(np.mean([a.elapsed_time(c) for a, c in fwd_evs]))

        # per-stage breakdown inside the step: a second capture of the same step with an
        # event at every boundary between C-ABI calls, so each call is timed where it runs
        # (inputs as the step leaves them, launch overlap inside a call kept, no graph
        # start); the events keep consecutive calls from overlapping, so the stages sum
        # to a little more than ms_per_step
        sev = [StepEvent() for _ in range(8)]
        sgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(sgraph, stream=st):
            step(evs=sev)
        torch.cuda.synchronize(dev)
        n_stage = max(3, min(args.steps, 10))
        per = np.zeros((n_stage, 7))
        for i in range(n_stage):
            flush_l2()
            sgraph.replay()
            st.synchronize()
            per[i] = [sev[j].elapsed_ms(sev[j + 1]) for j in range(7)]
        stage_ms = per.mean(0)
        eager_evs = [[ev() for _ in range(8)] for _ in range(n_stage)]
        for i in range(n_stage):
            flush_l2()
            step(eager_evs[i])
        torch.cuda.synchronize(dev)
        eager_ms = float(np.mean([e_[0].elapsed_time(e_[7]) for e_ in eager_evs]))

        # end to end through the public API: pinned host inputs in, results out
        x_h = x.cpu().pin_memory()
        dout_h = dout.cpu().pin_memory()
        out_h = torch.empty_like(L.out, device="cpu").pin_memory()
        dx_h = torch.empty_like(L.out, device="cpu").pin_memory()
        x_d = torch.empty_like(x)
        dout_d = torch.empty_like(dout)
        cs = torch.cuda.Stream(dev)       # copies that overlap compute: dout in, out back
        torch.cuda.synchronize(dev)
        e2e = []
        for i in range(args.steps):
            flush_l2()
            e0, e1 = ev(), ev()
            ev_dout, ev_fwd, ev_out = ev(), ev(), ev()
            e0.record(st)
            x_d.copy_(x_h, non_blocking=True)
            cs.wait_event(e0)
            with torch.cuda.stream(cs):
                dout_d.copy_(dout_h, non_blocking=True)   # during the forward
                ev_dout.record(cs)
            L.forward(x_d, Wr, Wu, Wd, W_gate=Wg, bias=b, noise=nz, token_mask=mk, stream=st,
                      shared=shared_w)
            ev_fwd.record(st)
            cs.wait_event(ev_fwd)
            with torch.cuda.stream(cs):
                out_h.copy_(L.out, non_blocking=True)     # during the backward
                ev_out.record(cs)
            st.wait_event(ev_dout)
            gg = L.backward(dout_d, stream=st)
            dx_h.copy_(gg["dx"], non_blocking=True)
            st.wait_event(ev_out)
            e1.record(st)
            e2e.append((e0, e1))
        torch.cuda.synchronize(dev)
        e2e_ms = float(np.mean([a.elapsed_time(c) for a, c in e2e]))

    # max over ranks
    ms, fwd_ms, e2e_ms, gemm_ms = max_over_ranks([ms_local, fwd_ms, e2e_ms, gemm_ms_local], dev,
                                                 world)
    if rank == 0:
        peaks, src = load_peaks()
        gemm_flop = work["gemm_fwd_flop"] + work["gemm_bwd_flop"]
        achieved = gemm_flop / (gemm_ms * 1e-3) / 1e12
        timed_region_s = args.steps * ms * 1e-3
        peak, kind = pick_bf16_peak(peaks, timed_region_s)
        traffic = gemm_traffic_from_profile(w.name)
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            cpu = cpu_baseline_leg(w, v, inp, args.seed, args.cpu_budget_s, args.one_core_budget_s)
        tok = job_rate(w.T, world, ms)
        es = 2 if dt == "bf16" else 4
        A = w.T * w.k
        line = {
            "metric": METRIC, "value": tok, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": dt, "data": "synthetic (seeded normals, random-init weights)",
            "config": workload_config(w, v),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak,
                         "traffic": traffic,
                         "traffic_scope": "ncu dram__bytes_read.sum + dram__bytes_write.sum over "
                                          "the grouped-GEMM launches of one step (one-pass capture)",
                         "kernel": "tc_grouped_gemm_kernel (all grouped-GEMM launches of a step)",
                         "timing": "external CUDA events around the two grouped-GEMM calls inside "
                                   "the replayed step graph (the timed steps themselves)",
                         "gemm_ms_per_step": gemm_ms,
                         "peak_source": f"{src} bf16 {kind} (timed region {timed_region_s:.2f} s)"},
            "cpu_baseline": cpu,
            "e2e": {"value": job_rate(w.T, world, e2e_ms), "unit": "tokens/s",
                    "h2d_bytes_per_step": (x.numel() + dout.numel()) * es,
                    "d2h_bytes_per_step": 2 * L.out.numel() * es},
            "clocks": clocks,
            "gpu_launches": int(launches_per_step * args.steps),
            "launches_per_step": int(launches_per_step),
            "eager_ms_per_step": eager_ms,
            "fwd_tokens_per_s": job_rate(w.T, world, fwd_ms),
            "stages_timing": "events between the C-ABI calls inside one replayed step graph "
                             "(L2 flushed before the step)",
            "stages_ms": {n: float(v_) for n, v_ in zip(
                ["route", "permute", "grouped_ffn", "combine", "combine_bwd", "grouped_ffn_bwd",
                 "router_bwd"], stage_ms)},
            "hbm_gbs": {"route": work["route_bytes"] / (stage_ms[0] * 1e-3) / 1e9,
                        "permute": work["permute_bytes"] / (stage_ms[1] * 1e-3) / 1e9,
                        "combine": work["combine_bytes"] / (stage_ms[3] * 1e-3) / 1e9,
                        "peak": peaks["hbm_gbs"]},
            "gemm_tflops": {"fwd": work["gemm_fwd_flop"] / (stage_ms[2] * 1e-3) / 1e12,
                            "bwd": work["gemm_bwd_flop"] / (stage_ms[5] * 1e-3) / 1e12},
            "routing": {"kept_assignments": A_kept, "dropped_assignments": int(stats[4]),
                        "drop_rate": stats[4] / A, "max_over_mean_kept": stats[5],
                        "max_over_mean_count": stats[7], "count_cv": stats[6],
                        "aux_loss": stats[0], "aux_switch": stats[1]},
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--ref-budget-s", type=float, default=3.0,
                    help="CPU seconds per reference-arm step")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0,
                    help="CPU seconds of the cpu_baseline sample (all host cores)")
    ap.add_argument("--one-core-budget-s", type=float, default=8.0,
                    help="CPU seconds of the one-core oracle sample (0: skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--f-shared", type=int, default=0,
                    help="add shared experts: a dense FFN of this hidden width on every token")
    ap.add_argument("--experts", type=int, default=0, help="override the workload's expert count")
    ap.add_argument("--top-k", type=int, default=0, help="override the workload's top-k")
    ap.add_argument("--temperature", type=float, default=1.0, help="router softmax temperature")
    ap.add_argument("--raw-gates", action="store_true",
                    help="gates = softmax probabilities of the selected experts (no renormalising)")
    ap.add_argument("--padding-mask", action="store_true",
                    help="right-padded sequences of 128 tokens: padding tokens select no expert")
    ap.add_argument("--straight-through", action="store_true",
                    help="Gumbel top-k selection, gates 1, straight-through router gradient")
    args = ap.parse_args(argv)
    w = moe_inputs.get(args.workload)
    if args.experts:
        w = replace(w, E=args.experts, name=f"{w.name}+E{args.experts}")
    if args.top_k:
        w = replace(w, k=args.top_k, name=f"{w.name}+k{args.top_k}")
    if args.f_shared:
        w = replace(w, f_shared=args.f_shared, name=f"{w.name}+shared{args.f_shared}")
    tags = ([f"tau{args.temperature:g}"] if args.temperature != 1.0 else []) + \
           (["rawgates"] if args.raw_gates else []) + (["mask"] if args.padding_mask else []) + \
           (["gumbelST"] if args.straight_through else [])
    if tags:
        w = replace(w, name=w.name + "+" + "+".join(tags))
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
