"""The no-allocation router entry point (moe_route_noalloc) against moe_route.

Some callers cannot allocate device memory -- a host framework that owns all
device memory through its own pool and forbids side allocations once running,
or a latency path that cannot afford cudaMalloc's cost and implicit
synchronisation -- so they cannot pass moe_route a workspace.
moe_route_noalloc takes its scratch from a static device array instead.  This
file is collected last so that a stop-at-first-failure run has already run
every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import moe_inputs
import top_routing_expert_moe_gb300 as moe
from tests import parity

pytestmark = pytest.mark.gpu


def _route_both(w, seed):
    """Route the same inputs through moe_route (caller workspace) and through
    moe_route_noalloc (static scratch); return both sets of outputs."""
    cfg = parity.gpu_cfg(w)
    inp = moe_inputs.make_inputs(w, seed, parts=("x", "W_r", "bias", "noise"))
    x = parity.to_torch(inp["x"], w.dtype)
    Wr = parity.to_torch(inp["W_r"], w.dtype)
    b = parity.to_torch(inp["bias"], "fp32")
    nz = parity.to_torch(inp["noise"], "fp32")
    dev = x.device

    def outputs():
        return dict(logits=torch.empty(w.T, w.E, dtype=torch.float32, device=dev),
                    topk=torch.empty(w.T, w.k, dtype=torch.int32, device=dev),
                    gate=torch.empty(w.T, w.k, dtype=torch.float32, device=dev),
                    counts=torch.empty(w.E, dtype=torch.int32, device=dev),
                    stats=torch.empty(9 + w.E, dtype=torch.float32, device=dev))

    ref = outputs()
    ws = torch.empty(moe.workspace_size(cfg), dtype=torch.uint8, device=dev)
    moe.moe_route(cfg, x, Wr, b, nz, None, ref["logits"], ref["topk"], ref["gate"], ref["counts"],
                  ref["stats"], ws)
    got = outputs()
    moe.moe_route_noalloc(cfg, x, Wr, b, nz, None, got["logits"], got["topk"], got["gate"],
                          got["counts"], got["stats"])
    torch.cuda.synchronize()
    return ref, got


def _check_same(ref, got):
    # the same kernels on the same inputs: every output byte for byte
    for key in ("logits", "topk", "gate", "counts", "stats"):
        assert torch.equal(got[key], ref[key]), key


def test_route_noalloc_matches_route_on_two_calls_in_a_row():
    # first call: the bf16 LLaMA4-style shape (gate noise), reduced tokens
    w1 = moe_inputs.get("llama4_bf16").with_tokens(4096)
    ref1, got1 = _route_both(w1, seed=5)
    _check_same(ref1, got1)
    # second call right after, on other inputs and another shape: the scratch
    # left by the first call must not leak into the result
    w2 = moe_inputs.get("skewed16_bf16").with_tokens(2048)
    ref2, got2 = _route_both(w2, seed=6)
    _check_same(ref2, got2)
    assert moe.last_device_status() == 0


def test_route_noalloc_rejects_configs_beyond_its_scratch():
    # E_pad * d bf16 transposed router weights alone exceed the static array
    cfg = moe.MoEConfig(T=128, d=16384, f=128, E=64, k=2)
    dev = torch.device("cuda")
    x = torch.zeros(cfg.T, cfg.d, dtype=torch.bfloat16, device=dev)
    Wr = torch.zeros(cfg.d, cfg.E, dtype=torch.bfloat16, device=dev)
    logits = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=dev)
    topk = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=dev)
    gate = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=dev)
    counts = torch.empty(cfg.E, dtype=torch.int32, device=dev)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_route_noalloc(cfg, x, Wr, None, None, None, logits, topk, gate, counts, None)
    assert ei.value.code == moe.ERR_SCRATCH_LIMIT
