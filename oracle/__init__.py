"""fp64 CPU oracle of the sparse MoE layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  It shares
no code with the CUDA library and never imports it.

The arithmetic lives in ``moe_oracle.c`` (plain loops, fp64), built with gcc
into ``oracle/_build/liboracle.so``.  This module only marshals numpy arrays.
``bruteforce.py`` is a second, independent restatement (per-expert mask loop)
used to pin the C oracle on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")

# statistics layout (see moe_oracle.c, OST_*)
ST_AUX_LOSS, ST_AUX_SWITCH, ST_ENTROPY, ST_NONFINITE = 0, 1, 2, 3
ST_DROPPED, ST_MAX_OVER_MEAN_KEPT, ST_COUNT_CV, ST_MAX_OVER_MEAN_COUNT = 4, 5, 6, 7
ST_TOKENS, ST_PBAR = 8, 9


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, OpenMP over independent loops)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d", ctypes.c_int), ("f", ctypes.c_int),
                ("E", ctypes.c_int), ("k", ctypes.c_int),
                ("capacity_factor", ctypes.c_double), ("swiglu", ctypes.c_int),
                ("normalize_gates", ctypes.c_int), ("aux_coef", ctypes.c_double),
                ("pad_m", ctypes.c_int), ("temperature", ctypes.c_double),
                ("straight_through", ctypes.c_int), ("f_shared", ctypes.c_int)]


@dataclass
class OracleConfig:
    T: int
    d: int
    f: int
    E: int
    k: int
    capacity_factor: float = 0.0   # <= 0 : no limit; pass the fp32 value the GPU sees
    swiglu: bool = False
    normalize_gates: bool = True
    aux_coef: float = 0.0
    pad_m: int = 1
    temperature: float = 1.0       # softmax temperature tau; pass the fp32 value the GPU sees
    straight_through: bool = False  # Gumbel top-k: select on logits + noise, gates 1
    f_shared: int = 0              # hidden width of the shared experts' FFN (0: none)

    def c(self) -> _Cfg:
        return _Cfg(self.T, self.d, self.f, self.E, self.k, float(self.capacity_factor),
                    int(self.swiglu), int(self.normalize_gates), float(self.aux_coef),
                    int(self.pad_m), float(self.temperature), int(self.straight_through),
                    int(self.f_shared))


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        _lib.oracle_capacity.restype = ctypes.c_int
        _lib.oracle_max_threads.restype = ctypes.c_int
        _lib.oracle_set_threads.restype = None
        _lib.oracle_set_threads.argtypes = [ctypes.c_int]
        _lib.oracle_route.restype = ctypes.c_int
        for name in ("oracle_router_logits", "oracle_permute", "oracle_combine", "oracle_stats",
                     "oracle_forward", "oracle_backward", "oracle_expert_apply",
                     "oracle_expert_forward", "oracle_shared_forward", "oracle_shared_add",
                     "oracle_expert_wgrad_entries"):
            getattr(_lib, name).restype = None
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _d(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def capacity(cfg: OracleConfig) -> int:
    return lib().oracle_capacity(ctypes.byref(cfg.c()))


def rows_bound(cfg: OracleConfig) -> int:
    return cfg.T * cfg.k + cfg.E * (cfg.pad_m - 1)


def router_logits(cfg, x, Wr, bias=None, noise=None):
    x, Wr, bias, noise = _d(x), _d(Wr), _d(bias), _d(noise)
    out = np.empty((cfg.T, cfg.E), np.float64)
    lib().oracle_router_logits(ctypes.byref(cfg.c()), _p(x), _p(Wr), _p(bias), _p(noise), _p(out))
    return out


def _mask(mask):
    return None if mask is None else np.ascontiguousarray(mask, np.uint8)


def route(cfg, logits, noise=None, mask=None):
    """Steps 2-4 on given logits.  ``noise`` is the selection noise of the
    straight-through mode; ``mask`` (uint8 [T], 0 = padding) may be None."""
    logits = _d(logits)
    noise, mask = _d(noise), _mask(mask)
    probs = np.empty((cfg.T, cfg.E), np.float64)
    topk = np.empty((cfg.T, cfg.k), np.int32)
    gate = np.empty((cfg.T, cfg.k), np.float64)
    counts = np.empty(cfg.E, np.int32)
    nf = lib().oracle_route(ctypes.byref(cfg.c()), _p(logits), _p(noise), _p(mask), _p(probs),
                            _p(topk), _p(gate), _p(counts))
    return dict(probs=probs, topk_idx=topk, gate=gate, counts=counts, nonfinite=nf)


def permute(cfg, topk_idx):
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    kept = np.empty(cfg.E, np.int32)
    offsets = np.empty(cfg.E + 1, np.int32)
    perm = np.empty(rows_bound(cfg), np.int32)
    slot = np.empty((cfg.T, cfg.k), np.int32)
    lib().oracle_permute(ctypes.byref(cfg.c()), _p(topk_idx), _p(kept), _p(offsets), _p(perm), _p(slot))
    return dict(kept=kept, offsets=offsets, perm_token=perm[:offsets[-1]].copy(), slot_of=slot)


def stats(cfg, probs, topk_idx, counts, kept, nonfinite=0):
    """Step 9 statistics (layout ST_*) from routed probabilities and counts."""
    out = np.empty(9 + cfg.E)
    lib().oracle_stats(ctypes.byref(cfg.c()), _p(_d(probs)),
                       _p(np.ascontiguousarray(topk_idx, np.int32)),
                       _p(np.ascontiguousarray(counts, np.int32)),
                       _p(np.ascontiguousarray(kept, np.int32)), ctypes.c_int(int(nonfinite)),
                       _p(out))
    return out


def expert_apply(cfg, e, x_row, Wup, Wgate, Wdown):
    y = np.empty(cfg.d, np.float64)
    lib().oracle_expert_apply(ctypes.byref(cfg.c()), int(e), _p(_d(x_row)), _p(_d(Wup)),
                              _p(_d(Wgate) if cfg.swiglu else None), _p(_d(Wdown)), _p(y))
    return y


def expert_forward(cfg, e, x_row, Wup, Wdown, Wgate=None):
    """One expert on one token: dict(h, u, act, y) (h is g for SwiGLU; u None for SiLU)."""
    f, d = cfg.f, cfg.d
    h, act, y = np.empty(f), np.empty(f), np.empty(d)
    u = np.empty(f) if cfg.swiglu else None
    lib().oracle_expert_forward(ctypes.byref(cfg.c()), int(e), _p(_d(x_row)), _p(_d(Wup)),
                                _p(_d(Wgate) if cfg.swiglu else None), _p(_d(Wdown)), _p(h),
                                _p(u), _p(act), _p(y))
    return dict(h=h, u=u, act=act, y=y)


def shared_forward(cfg, x_row, Wup_s, Wdown_s, Wgate_s=None):
    """The shared experts' FFN on one token: dict(h, u, act, y) (width f_shared)."""
    fs, d = cfg.f_shared, cfg.d
    h, act, y = np.empty(fs), np.empty(fs), np.empty(d)
    u = np.empty(fs) if cfg.swiglu else None
    lib().oracle_shared_forward(ctypes.byref(cfg.c()), _p(_d(x_row)), _p(_d(Wup_s)),
                                _p(_d(Wgate_s) if cfg.swiglu else None), _p(_d(Wdown_s)), _p(h),
                                _p(u), _p(act), _p(y))
    return dict(h=h, u=u, act=act, y=y)


def _shared_args(cfg, Wup_s, Wgate_s, Wdown_s):
    if cfg.f_shared <= 0:
        return None, None, None
    if Wup_s is None or Wdown_s is None or (cfg.swiglu and Wgate_s is None):
        raise ValueError("f_shared > 0 needs the shared experts' weights")
    return _d(Wup_s), _d(Wgate_s) if cfg.swiglu else None, _d(Wdown_s)


def forward(cfg, x, Wr, Wup, Wdown, Wgate=None, bias=None, noise=None, logits_in=None, mask=None,
            Wup_s=None, Wdown_s=None, Wgate_s=None):
    """Steps 1-9. ``logits_in`` (e.g. the GPU's fp32 logits) replaces step 1.
    With ``cfg.f_shared > 0`` the shared experts' FFN (weights ``*_s``) joins
    every token's output with weight 1."""
    Wus, Wgs, Wds = _shared_args(cfg, Wup_s, Wgate_s, Wdown_s)
    x, Wr, Wup, Wdown, Wgate = _d(x), _d(Wr), _d(Wup), _d(Wdown), _d(Wgate)
    bias, noise, logits_in, mask = _d(bias), _d(noise), _d(logits_in), _mask(mask)
    T, E, k, d = cfg.T, cfg.E, cfg.k, cfg.d
    r = dict(logits=np.empty((T, E)), probs=np.empty((T, E)), topk_idx=np.empty((T, k), np.int32),
             gate=np.empty((T, k)), counts=np.empty(E, np.int32), kept=np.empty(E, np.int32),
             offsets=np.empty(E + 1, np.int32), perm_token=np.empty(rows_bound(cfg), np.int32),
             slot_of=np.empty((T, k), np.int32), out=np.empty((T, d)), stats=np.empty(9 + E))
    lib().oracle_forward(ctypes.byref(cfg.c()), _p(x), _p(Wr), _p(bias), _p(noise), _p(mask), _p(Wup),
                         _p(Wgate), _p(Wdown), _p(logits_in),
                         *[_p(r[n]) for n in ("logits", "probs", "topk_idx", "gate", "counts", "kept",
                                               "offsets", "perm_token", "slot_of", "out", "stats")],
                         _p(Wus), _p(Wgs), _p(Wds))
    r["perm_token"] = r["perm_token"][: r["offsets"][-1]].copy()
    return r


def backward(cfg, x, Wr, Wup, Wdown, logits, topk_idx, gate, slot_of, dout, Wgate=None,
             with_bias=False, per_slot=False, pbar=None, T_aux=0, Wup_s=None, Wdown_s=None,
             Wgate_s=None):
    """Step 10: gradients of <dout, out> + aux loss (written, not accumulated).
    For a sample of a larger batch pass that batch's ``pbar`` and ``T_aux``.
    With shared experts the result also holds dWup_s, dWgate_s, dWdown_s."""
    Wus, Wgs, Wds = _shared_args(cfg, Wup_s, Wgate_s, Wdown_s)
    x, Wr, Wup, Wdown, Wgate = _d(x), _d(Wr), _d(Wup), _d(Wdown), _d(Wgate)
    logits, gate, dout = _d(logits), _d(gate), _d(dout)
    topk_idx = np.ascontiguousarray(topk_idx, np.int32)
    slot_of = np.ascontiguousarray(slot_of, np.int32)
    T, E, k, d, f = cfg.T, cfg.E, cfg.k, cfg.d, cfg.f
    g = dict(dx=np.empty((T, d)), dWr=np.empty((d, E)), db=np.empty(E) if with_bias else None,
             dWup=np.empty((E, d, f)), dWgate=np.empty((E, d, f)) if cfg.swiglu else None,
             dWdown=np.empty((E, f, d)), dgate=np.empty((T, k)), dlogits=np.empty((T, E)),
             dh_slot=np.empty((T, k, 2 if cfg.swiglu else 1, f)) if per_slot else None,
             dxp_slot=np.empty((T, k, d)) if per_slot else None)
    fs = cfg.f_shared
    if fs > 0:
        g.update(dWup_s=np.empty((d, fs)), dWgate_s=np.empty((d, fs)) if cfg.swiglu else None,
                 dWdown_s=np.empty((fs, d)))
    lib().oracle_backward(ctypes.byref(cfg.c()), _p(x), _p(Wr), _p(Wup), _p(Wgate), _p(Wdown),
                          _p(logits), _p(topk_idx), _p(gate), _p(slot_of), _p(dout),
                          *[_p(g[n]) for n in ("dx", "dWr", "db", "dWup", "dWgate", "dWdown",
                                               "dgate", "dlogits", "dh_slot", "dxp_slot")],
                          _p(_d(pbar)), ctypes.c_int(int(T_aux)),
                          _p(Wus), _p(Wgs), _p(Wds),
                          *[_p(g.get(n)) for n in ("dWup_s", "dWgate_s", "dWdown_s")])
    return g


WGRAD_DOWN, WGRAD_UP, WGRAD_GATE = 0, 1, 2


def expert_wgrad_entries(cfg, xs, gates, douts, Wu_e, Wd_e, which, rows, cols, Wg_e=None):
    """Single entries of one expert's weight gradients from their definition:
    which[q] = WGRAD_DOWN -> dW_down[rows[q], cols[q]], WGRAD_UP -> dW_up[...],
    WGRAD_GATE -> dW_gate[...] (SwiGLU).  xs / douts [n, d] are the inputs and
    output gradients of the expert's kept tokens (ascending), gates [n] their
    gates; Wu_e, Wg_e [d, f] and Wd_e [f, d] the expert's weight blocks."""
    xs, douts, gates = _d(xs), _d(douts), _d(gates)
    n = len(gates)
    assert xs.shape == (n, cfg.d) and douts.shape == (n, cfg.d)
    which = np.ascontiguousarray(which, np.int32)
    rows = np.ascontiguousarray(rows, np.int32)
    cols = np.ascontiguousarray(cols, np.int32)
    out = np.empty(len(which), np.float64)
    lib().oracle_expert_wgrad_entries(ctypes.byref(cfg.c()), ctypes.c_int(n), _p(xs), _p(gates),
                                      _p(douts), _p(_d(Wu_e)),
                                      _p(_d(Wg_e) if cfg.swiglu else None), _p(_d(Wd_e)),
                                      ctypes.c_int(len(which)), _p(which), _p(rows), _p(cols),
                                      _p(out))
    return out


def max_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(lib().oracle_max_threads())


def set_threads(n: int) -> None:
    """Set the OpenMP thread count of later oracle calls from this thread."""
    lib().oracle_set_threads(int(n))
