"""Failure detection on the device without a GPU fault: a bounded wait that
runs out records MOE_ERR_TIMEOUT, the kernel returns, and the context stays
usable for the next layer call."""
import time

import pytest
import torch

import moe_inputs
import top_routing_expert_moe_gb300 as moe
from tests import parity

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout():
    assert moe.last_device_status() == 0
    t0 = time.time()
    moe.selftest_bounded_wait(20_000_000)          # 20 ms on a barrier nobody arrives on
    assert moe.last_device_status() == moe.ERR_TIMEOUT
    assert time.time() - t0 < 5.0
    assert moe.last_device_status() == 0           # reading cleared it
    # the context is still usable: a small layer runs and matches the oracle
    w = moe_inputs.get("small_bf16").with_tokens(256)
    from dataclasses import replace
    w = replace(w, d=256, f=256)
    rep, _ = parity.full_check(w, moe_inputs.make_inputs(w, 0))
    assert rep["out_rel"] < parity.TOL["bf16"]


def test_selftest_rejects_out_of_range_limits():
    with pytest.raises(moe.MoEError):
        moe.selftest_bounded_wait(0)
    with pytest.raises(moe.MoEError):
        moe.selftest_bounded_wait(2_000_000_000)
    torch.cuda.synchronize()


def test_tma_kernels_skip_work_while_a_timeout_is_pending():
    """Fail fast: after a bounded wait ran out and before the host reads the
    status, the router and grouped-GEMM kernels skip their work (so a lost
    arrival costs one time limit, not one per launch).  Their outputs keep the
    sentinel they were filled with, the status still reads MOE_ERR_TIMEOUT, and
    once it has been read the next call matches the oracle again."""
    from dataclasses import replace
    assert moe.last_device_status() == 0
    moe.selftest_bounded_wait(20_000_000)
    torch.cuda.synchronize()                       # recorded, not read
    w = replace(moe_inputs.get("small_bf16").with_tokens(256), d=256, f=256)
    inp = moe_inputs.make_inputs(w, 0)
    cfg = parity.gpu_cfg(w)
    L = moe.MoELayer(cfg)
    L.logits.fill_(-7.0)
    L.h_saved.fill_(3.0)
    L.y_perm.fill_(5.0)
    t0 = time.time()
    L.forward(parity.to_torch(inp["x"], "bf16"), parity.to_torch(inp["W_r"], "bf16"),
              parity.to_torch(inp["W_up"], "bf16"), parity.to_torch(inp["W_down"], "bf16"))
    torch.cuda.synchronize()
    assert time.time() - t0 < 3.0
    assert (L.logits == -7.0).all(), "the router ran although a timeout was pending"
    assert (L.h_saved == 3.0).all() and (L.y_perm == 5.0).all(), "a grouped GEMM ran"
    assert moe.last_device_status() == moe.ERR_TIMEOUT
    assert moe.last_device_status() == 0
    rep, _ = parity.full_check(w, inp)
    assert rep["out_rel"] < parity.TOL["bf16"]
