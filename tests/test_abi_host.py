"""Host-side checks of the C ABI: the library builds, loads, exports every
symbol include/moe.h declares, and validates arguments -- no GPU calls."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import top_routing_expert_moe_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)))


def test_header_declares_the_layer_entry_points():
    names = declared_symbols()
    for n in ("moe_route", "moe_permute", "moe_grouped_ffn", "moe_combine", "moe_backward",
              "moe_workspace_size", "moe_error_string", "moe_last_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = moe.load_library()
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def declared_param_counts():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    out = {}
    for m in re.finditer(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(([^)]*)\)", src):
        params = [p for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        out[m.group(1)] = len(params)
    return out


def test_binding_signatures_match_header():
    lib = moe.load_library()
    counts = declared_param_counts()
    for name, n in counts.items():
        argtypes = getattr(lib, name).argtypes
        assert argtypes is not None and len(argtypes) == n, (name, n, argtypes and len(argtypes))


def test_struct_layout_matches_header():
    # 14 four-byte fields, no padding
    assert ctypes.sizeof(moe.MoEConfig) == 56
    assert ctypes.sizeof(moe.MoESharedFFN) == 13 * 8


def test_config_validation():
    ok = moe.MoEConfig(T=2048, d=1024, f=2048, E=4, k=2, capacity_factor=1.2)
    assert moe.check_config(ok) == moe.OK
    bad = [dict(T=0), dict(k=5), dict(E=0), dict(pad_m=0), dict(dtype=7), dict(ffn=3),
           dict(normalize_gates=2), dict(capacity_factor=float("nan")),
           dict(temperature=float("nan")), dict(temperature=-1.0), dict(temperature=float("inf")),
           dict(straight_through=2), dict(f_shared=-128)]
    for b in bad:
        kw = dict(T=64, d=256, f=256, E=4, k=2)
        kw.update(b)
        assert moe.check_config(moe.MoEConfig(**kw)) == moe.ERR_INVALID_ARG, b
    unsup = [dict(E=65, k=2), dict(k=9, E=16), dict(d=200), dict(f=136), dict(pad_m=64),
             dict(f_shared=200)]
    for b in unsup:
        kw = dict(T=64, d=256, f=256, E=4, k=2)
        kw.update(b)
        assert moe.check_config(moe.MoEConfig(**kw)) == moe.ERR_UNSUPPORTED, b
    # fp32 accepts any multiple-of-8 width and any padding
    assert moe.check_config(moe.MoEConfig(T=5, d=24, f=40, E=3, k=2, dtype=moe.F32, pad_m=1)) == 0


@pytest.mark.parametrize("T,E,k,cf", [(2048, 4, 2, 1.2), (16384, 8, 2, 1.2), (65536, 16, 2, 1.2),
                                      (77, 4, 2, 0.0), (10, 2, 2, 50.0), (999, 7, 3, 0.37),
                                      (5, 5, 5, 1.0)])
def test_capacity_matches_oracle(T, E, k, cf):
    c = moe.MoEConfig(T=T, d=8, f=8, E=E, k=k, capacity_factor=cf, dtype=moe.F32, pad_m=1)
    want = oracle.capacity(oracle.OracleConfig(T=T, d=8, f=8, E=E, k=k,
                                               capacity_factor=float(np.float32(cf))))
    assert moe.capacity(c) == want


def test_rows_capacity_and_workspace():
    c = moe.MoEConfig(T=2048, d=1024, f=2048, E=4, k=2, capacity_factor=1.2)
    # min(T k, E C) + E (pad - 1) = min(4096, 4*1229) + 4*127
    assert moe.rows_capacity(c) == 4096 + 4 * 127
    assert moe.workspace_size(c) >= (4096 + 508) * 1024 * 2 * 3


def test_null_and_misaligned_pointers_are_rejected_before_launch():
    lib = moe.load_library()
    c = moe.MoEConfig(T=64, d=256, f=256, E=4, k=2)
    args = [ctypes.byref(c)] + [None] * 11 + [None]
    assert lib.moe_route(*args) == moe.ERR_INVALID_ARG
    p = ctypes.c_void_p(0x1000 + 8)  # misaligned
    args = [ctypes.byref(c)] + [p] * 11 + [None]
    assert lib.moe_route(*args) == moe.ERR_INVALID_ARG
    assert lib.moe_combine(ctypes.byref(c), None, None, None, None, None, None) == moe.ERR_INVALID_ARG
    assert lib.moe_route(None, *([None] * 12)) == moe.ERR_INVALID_ARG


def test_error_strings():
    for code in range(-7, 1):
        assert moe.error_string(code)
    assert moe.error_string(-99) == "unknown status"


def test_shared_rows_and_block_presence_checks():
    c = moe.MoEConfig(T=333, d=256, f=256, E=4, k=2, f_shared=384)
    assert moe.shared_rows(c) == 384                      # T rounded up to 128 (bf16)
    assert moe.shared_rows(moe.MoEConfig(T=333, d=256, f=256, E=4, k=2)) == 0
    assert moe.shared_rows(moe.MoEConfig(T=97, d=64, f=96, E=4, k=2, dtype=moe.F32,
                                         pad_m=1, f_shared=40)) == 97
    # the workspace covers the shared FFN's backward intermediates
    assert moe.workspace_size(c) > moe.workspace_size(moe.MoEConfig(T=333, d=256, f=256, E=4, k=2))
    lib = moe.load_library()
    p = ctypes.c_void_p(0x10000)                          # aligned, never dereferenced
    # f_shared > 0 needs the block; f_shared = 0 forbids it (checked before any launch)
    assert lib.moe_combine(ctypes.byref(c), p, p, p, None, p, None) == moe.ERR_INVALID_ARG
    c0 = moe.MoEConfig(T=333, d=256, f=256, E=4, k=2)
    blk = moe.MoESharedFFN()
    assert lib.moe_combine(ctypes.byref(c0), p, p, p, ctypes.byref(blk), p, None) == \
        moe.ERR_INVALID_ARG
    # a block missing the field moe_combine reads
    assert lib.moe_combine(ctypes.byref(c), p, p, p, ctypes.byref(blk), p, None) == \
        moe.ERR_INVALID_ARG
