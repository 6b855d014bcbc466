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
