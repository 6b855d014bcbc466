"""GB300 (sm_103a) sparse MoE layer: Python binding of the C ABI in include/moe.h.

Argument marshalling only: every step of the layer runs in the CUDA kernels of
``libmoe.so``.  Tensors are torch CUDA tensors (torch supplies device memory
and streams); each function mirrors the C entry point of the same name.  If
the library is missing the import of any entry point raises -- there is no
CPU fallback.

    import top_routing_expert_moe_gb300 as moe
    cfg = moe.MoEConfig(T=2048, d=1024, f=2048, E=4, k=2, capacity_factor=1.2,
                        dtype=moe.BF16)
    layer = moe.MoELayer(cfg, device="cuda")
    out = layer.forward(x, W_r, W_up, W_down)
    grads = layer.backward(dout)
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

F32, BF16 = 0, 1
SILU, SWIGLU = 0, 1
STAT_AUX_LOSS, STAT_AUX_SWITCH, STAT_ENTROPY, STAT_NONFINITE = 0, 1, 2, 3
STAT_DROPPED, STAT_MAX_OVER_MEAN_KEPT, STAT_COUNT_CV, STAT_MAX_OVER_MEAN_COUNT = 4, 5, 6, 7
STAT_TOKENS, STAT_PBAR = 8, 9

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_NONFINITE, ERR_DEVICE_BOUNDS = \
    0, -1, -2, -3, -4, -5, -6
ERR_SCRATCH_LIMIT = -7
ROUTE_NOALLOC_SCRATCH_BYTES = 2 * 1024 * 1024


class MoEConfig(ctypes.Structure):
    """Mirror of ``moe_config`` (include/moe.h)."""
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("f", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float), ("ffn", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("normalize_gates", ctypes.c_int32),
                ("aux_coef", ctypes.c_float), ("pad_m", ctypes.c_int32),
                ("temperature", ctypes.c_float), ("straight_through", ctypes.c_int32),
                ("f_shared", ctypes.c_int32)]

    def __init__(self, T, d, f, E, k, capacity_factor=0.0, ffn=SILU, dtype=BF16,
                 normalize_gates=1, aux_coef=0.0, pad_m=128, temperature=1.0,
                 straight_through=0, f_shared=0):
        super().__init__(T, d, f, E, k, capacity_factor, ffn, dtype, normalize_gates, aux_coef,
                         pad_m, temperature, int(straight_through), int(f_shared))

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == BF16 else torch.float32

    @property
    def nh(self):
        return 2 if self.ffn == SWIGLU else 1

    def __repr__(self):
        return ("MoEConfig(" + ", ".join(f"{n}={getattr(self, n)!r}" for n, _ in self._fields_) + ")")


def config_for(shape, pad_m=128, normalize=True, temperature=1.0, straight_through=False):
    """A MoEConfig from a layer-shape record with fields T, d, f, E, k,
    capacity_factor, swiglu, dtype ("bf16" / "fp32"), aux_coef and f_shared
    (e.g. a seeded workload), plus the router options."""
    return MoEConfig(T=shape.T, d=shape.d, f=shape.f, E=shape.E, k=shape.k,
                     capacity_factor=shape.capacity_factor,
                     ffn=SWIGLU if shape.swiglu else SILU,
                     dtype=BF16 if shape.dtype == "bf16" else F32,
                     normalize_gates=1 if normalize else 0, aux_coef=shape.aux_coef, pad_m=pad_m,
                     temperature=temperature, straight_through=int(straight_through),
                     f_shared=shape.f_shared)


def tensor_from_numpy(a, dtype: str, device="cuda"):
    """Copy a host array to the device: bf16 tensors arrive as their uint16 bit
    patterns and are reinterpreted, everything else keeps its numpy dtype.
    None stays None."""
    if a is None:
        return None
    import numpy as np
    if dtype == "bf16" and a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


_SHARED_FIELDS = ("x", "W_up", "W_gate", "W_down", "h", "act", "y", "dout", "dh", "dx",
                  "dW_up", "dW_gate", "dW_down")


class MoESharedFFN(ctypes.Structure):
    """Mirror of ``moe_shared_ffn`` (include/moe.h): device pointers of the
    shared experts' FFN (weights, saved activations, gradients)."""
    _fields_ = [(n, ctypes.c_void_p) for n in _SHARED_FIELDS]


def shared_block(**tensors) -> MoESharedFFN:
    """A ``moe_shared_ffn`` from torch tensors given by field name (others NULL).
    The block holds references to the tensors, so their memory stays allocated
    for as long as the block (or a CUDA graph captured with it) is in use."""
    unknown = set(tensors) - set(_SHARED_FIELDS)
    if unknown:
        raise ValueError(f"unknown shared-expert fields {sorted(unknown)}")
    b = MoESharedFFN()
    for n, t in tensors.items():
        setattr(b, n, None if t is None else _p(t).value)
    b._tensors = dict(tensors)
    return b


def _sh(shared):
    return None if shared is None else ctypes.byref(shared)


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {error_string(code)} ({code})")


_lib = None
_SIGS = {
    "moe_check_config": [ctypes.c_void_p],
    "moe_capacity": [ctypes.c_void_p, ctypes.c_void_p],
    "moe_rows_capacity": [ctypes.c_void_p, ctypes.c_void_p],
    "moe_shared_rows": [ctypes.c_void_p, ctypes.c_void_p],
    "moe_workspace_size": [ctypes.c_void_p, ctypes.c_void_p],
    "moe_route": [ctypes.c_void_p] * 13,
    "moe_route_noalloc": [ctypes.c_void_p] * 12,
    "moe_permute": [ctypes.c_void_p] * 11,
    "moe_grouped_ffn": [ctypes.c_void_p] * 12,
    "moe_combine": [ctypes.c_void_p] * 7,
    "moe_combine_backward": [ctypes.c_void_p] * 10,
    "moe_grouped_ffn_backward": [ctypes.c_void_p] * 17,
    "moe_router_backward": [ctypes.c_void_p] * 17,
    "moe_backward": [ctypes.c_void_p] * 27,
    "moe_last_device_status": [ctypes.c_void_p, ctypes.c_void_p],
    "moe_selftest_bounded_wait": [ctypes.c_ulonglong, ctypes.c_void_p],
}


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libmoe.so (building it with nvcc when absent or stale)."""
    global _lib
    if _lib is None:
        path = _build.build() if build_if_missing else _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libmoe.so not found at {path}; run top_routing_expert_moe_gb300.build")
        lib = ctypes.CDLL(path)
        for name, argtypes in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = argtypes
            fn.restype = ctypes.c_int
        lib.moe_error_string.argtypes = [ctypes.c_int]
        lib.moe_error_string.restype = ctypes.c_char_p
        lib.moe_launch_count.argtypes = []
        lib.moe_launch_count.restype = ctypes.c_uint64
        _lib = lib
    return _lib


def error_string(code: int) -> str:
    return load_library().moe_error_string(int(code)).decode()


def _p(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("tensors passed to the MoE library must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _s(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _call(name, *args):
    rc = getattr(load_library(), name)(*args)
    if rc != 0:
        raise MoEError(rc, name)


# ----------------------------------------------------------------- host queries
def check_config(cfg: MoEConfig) -> int:
    return load_library().moe_check_config(ctypes.byref(cfg))


def capacity(cfg: MoEConfig) -> int:
    v = ctypes.c_int32()
    _call("moe_capacity", ctypes.byref(cfg), ctypes.byref(v))
    return v.value


def rows_capacity(cfg: MoEConfig) -> int:
    v = ctypes.c_int64()
    _call("moe_rows_capacity", ctypes.byref(cfg), ctypes.byref(v))
    return v.value


def shared_rows(cfg: MoEConfig) -> int:
    v = ctypes.c_int64()
    _call("moe_shared_rows", ctypes.byref(cfg), ctypes.byref(v))
    return v.value


def workspace_size(cfg: MoEConfig) -> int:
    v = ctypes.c_size_t()
    _call("moe_workspace_size", ctypes.byref(cfg), ctypes.byref(v))
    return v.value


def launch_count() -> int:
    return int(load_library().moe_launch_count())


def selftest_bounded_wait(limit_ns: int, stream=None) -> None:
    """Run the device-side timeout self-test (the status is read with
    last_device_status())."""
    _call("moe_selftest_bounded_wait", ctypes.c_ulonglong(int(limit_ns)), _s(stream))


def last_device_status(stream=None) -> int:
    v = ctypes.c_int()
    _call("moe_last_device_status", _s(stream), ctypes.byref(v))
    return v.value


# ----------------------------------------------------------------- entry points
def moe_route(cfg, x, W_r, bias, noise, token_mask, logits, topk_idx, gate, counts, stats, ws,
              stream=None):
    _call("moe_route", ctypes.byref(cfg), _p(x), _p(W_r), _p(bias), _p(noise), _p(token_mask),
          _p(logits), _p(topk_idx), _p(gate), _p(counts), _p(stats), _p(ws), _s(stream))


def moe_route_noalloc(cfg, x, W_r, bias, noise, token_mask, logits, topk_idx, gate, counts, stats,
                      stream=None):
    """moe_route without a workspace, for callers that cannot allocate device
    memory: scratch comes from the library's static device array (shared by all
    calls; overlapping calls race)."""
    _call("moe_route_noalloc", ctypes.byref(cfg), _p(x), _p(W_r), _p(bias), _p(noise),
          _p(token_mask), _p(logits), _p(topk_idx), _p(gate), _p(counts), _p(stats), _s(stream))


def moe_permute(cfg, x, topk_idx, x_perm, perm_token, slot_of, kept, offsets, stats, ws,
                stream=None):
    _call("moe_permute", ctypes.byref(cfg), _p(x), _p(topk_idx), _p(x_perm), _p(perm_token),
          _p(slot_of), _p(kept), _p(offsets), _p(stats), _p(ws), _s(stream))


def moe_grouped_ffn(cfg, x_perm, offsets, W_up, W_gate, W_down, h_saved, act, y_perm, ws,
                    stream=None, shared=None):
    _call("moe_grouped_ffn", ctypes.byref(cfg), _p(x_perm), _p(offsets), _p(W_up), _p(W_gate),
          _p(W_down), _p(h_saved), _p(act), _p(y_perm), _sh(shared), _p(ws), _s(stream))


def moe_combine(cfg, y_perm, slot_of, gate, out, stream=None, shared=None):
    _call("moe_combine", ctypes.byref(cfg), _p(y_perm), _p(slot_of), _p(gate), _sh(shared),
          _p(out), _s(stream))


def moe_combine_backward(cfg, dout, y_perm, gate, slot_of, perm_token, offsets, dy_perm, dgate,
                         stream=None):
    _call("moe_combine_backward", ctypes.byref(cfg), _p(dout), _p(y_perm), _p(gate), _p(slot_of),
          _p(perm_token), _p(offsets), _p(dy_perm), _p(dgate), _s(stream))


def moe_grouped_ffn_backward(cfg, x_perm, offsets, W_up, W_gate, W_down, h_saved, act, dy_perm,
                             dh, dx_perm, dW_up, dW_gate, dW_down, ws, stream=None, shared=None):
    _call("moe_grouped_ffn_backward", ctypes.byref(cfg), _p(x_perm), _p(offsets), _p(W_up),
          _p(W_gate), _p(W_down), _p(h_saved), _p(act), _p(dy_perm), _p(dh), _p(dx_perm),
          _p(dW_up), _p(dW_gate), _p(dW_down), _sh(shared), _p(ws), _s(stream))


def moe_router_backward(cfg, x, W_r, logits, topk_idx, gate, slot_of, dgate, dx_perm, stats, dx,
                        dW_r, dbias, dlogits, ws, stream=None, shared=None):
    _call("moe_router_backward", ctypes.byref(cfg), _p(x), _p(W_r), _p(logits), _p(topk_idx),
          _p(gate), _p(slot_of), _p(dgate), _p(dx_perm), _sh(shared), _p(stats), _p(dx),
          _p(dW_r), _p(dbias), _p(dlogits), _p(ws), _s(stream))


def moe_backward(cfg, x, W_r, W_up, W_gate, W_down, logits, topk_idx, gate, slot_of, perm_token,
                 offsets, x_perm, h_saved, act, y_perm, stats, dout, dx, dW_r, dbias, dW_up,
                 dW_gate, dW_down, ws, stream=None, shared=None):
    _call("moe_backward", ctypes.byref(cfg), _p(x), _p(W_r), _p(W_up), _p(W_gate), _p(W_down),
          _p(logits), _p(topk_idx), _p(gate), _p(slot_of), _p(perm_token), _p(offsets),
          _p(x_perm), _p(h_saved), _p(act), _p(y_perm), _p(stats), _p(dout), _p(dx), _p(dW_r),
          _p(dbias), _p(dW_up), _p(dW_gate), _p(dW_down), _sh(shared), _p(ws), _s(stream))


# ----------------------------------------------------------------- convenience layer
class MoELayer:
    """Owns the routing cache, permuted buffers and workspace of one layer
    configuration (all torch-allocated once) and chains the entry points.
    With cfg.f_shared > 0, forward() takes the shared experts' weights
    (``shared=(W_up_s, W_down_s, W_gate_s or None)``) and backward() also
    returns their gradients (dW_up_s, dW_gate_s, dW_down_s)."""

    def __init__(self, cfg: MoEConfig, device="cuda"):
        rc = check_config(cfg)
        if rc != 0:
            raise MoEError(rc, "moe_check_config")
        self.cfg = cfg
        dev = torch.device(device)
        dt = cfg.torch_dtype
        T, d, f, E, k = cfg.T, cfg.d, cfg.f, cfg.E, cfg.k
        self.rows_cap = R = rows_capacity(cfg)
        e = lambda *s, dtype=dt: torch.empty(*s, dtype=dtype, device=dev)  # noqa: E731
        self.logits = e(T, E, dtype=torch.float32)
        self.topk_idx = e(T, k, dtype=torch.int32)
        self.gate = e(T, k, dtype=torch.float32)
        self.counts = e(E, dtype=torch.int32)
        self.stats = e(9 + E, dtype=torch.float32)
        self.x_perm = e(R, d)
        self.perm_token = e(R, dtype=torch.int32)
        self.slot_of = e(T, k, dtype=torch.int32)
        self.kept = e(E, dtype=torch.int32)
        self.offsets = e(E + 1, dtype=torch.int32)
        self.h_saved = e(cfg.nh, R, f)
        self.act = e(R, f)
        self.y_perm = e(R, d)
        self.out = e(T, d)
        self.ws = e(max(workspace_size(cfg), 256), dtype=torch.uint8)
        self.shared_rows = Ts = shared_rows(cfg)
        if cfg.f_shared > 0:
            fs = cfg.f_shared
            self.h_shared = e(cfg.nh, Ts, fs)
            self.act_shared = e(Ts, fs)
            self.y_shared = e(Ts, d)
        self._grads = None
        self._inputs = None
        self._shared_w = None

    def _shared_fwd(self, x):
        if self.cfg.f_shared <= 0:
            return None
        Wu, Wd, Wg = self._shared_w
        return shared_block(x=x, W_up=Wu, W_gate=Wg, W_down=Wd, h=self.h_shared,
                            act=self.act_shared, y=self.y_shared)

    def forward(self, x, W_r, W_up, W_down, W_gate=None, bias=None, noise=None, token_mask=None,
                stream=None, shared=None):
        c = self.cfg
        if (c.f_shared > 0) != (shared is not None):
            raise ValueError("shared-expert weights are required iff cfg.f_shared > 0")
        if shared is not None:
            Wu_s, Wd_s = shared[0], shared[1]
            Wg_s = shared[2] if len(shared) > 2 else None
            self._shared_w = (Wu_s, Wd_s, Wg_s)
        sh = self._shared_fwd(x)
        moe_route(c, x, W_r, bias, noise, token_mask, self.logits, self.topk_idx, self.gate,
                  self.counts, self.stats, self.ws, stream)
        moe_permute(c, x, self.topk_idx, self.x_perm, self.perm_token, self.slot_of, self.kept,
                    self.offsets, self.stats, self.ws, stream)
        moe_grouped_ffn(c, self.x_perm, self.offsets, W_up, W_gate, W_down, self.h_saved,
                        self.act, self.y_perm, self.ws, stream, shared=sh)
        moe_combine(c, self.y_perm, self.slot_of, self.gate, self.out, stream, shared=sh)
        self._inputs = (x, W_r, W_up, W_gate, W_down, bias)
        return self.out

    def grads(self):
        if self._grads is None:
            c, dev = self.cfg, self.out.device
            dt = c.torch_dtype
            self._grads = dict(
                dx=torch.empty(c.T, c.d, dtype=dt, device=dev),
                dW_r=torch.empty(c.d, c.E, dtype=dt, device=dev),
                dbias=torch.empty(c.E, dtype=torch.float32, device=dev),
                dW_up=torch.empty(c.E, c.d, c.f, dtype=dt, device=dev),
                dW_gate=(torch.empty(c.E, c.d, c.f, dtype=dt, device=dev)
                         if c.ffn == SWIGLU else None),
                dW_down=torch.empty(c.E, c.f, c.d, dtype=dt, device=dev))
            if c.f_shared > 0:
                fs = c.f_shared
                self._grads.update(
                    dW_up_s=torch.empty(c.d, fs, dtype=dt, device=dev),
                    dW_gate_s=(torch.empty(c.d, fs, dtype=dt, device=dev)
                               if c.ffn == SWIGLU else None),
                    dW_down_s=torch.empty(fs, c.d, dtype=dt, device=dev))
        return self._grads

    def shared_block(self, dout=None, dh=None, dx=None):
        """The layer's moe_shared_ffn block (forward buffers, weights, gradient
        outputs; dout / dh / dx as given), or None without shared experts."""
        if self.cfg.f_shared <= 0:
            return None
        x = self._inputs[0]
        Wu, Wd, Wg = self._shared_w
        g = self.grads()
        return shared_block(x=x, W_up=Wu, W_gate=Wg, W_down=Wd, h=self.h_shared,
                            act=self.act_shared, y=self.y_shared, dout=dout, dh=dh, dx=dx,
                            dW_up=g["dW_up_s"], dW_gate=g["dW_gate_s"], dW_down=g["dW_down_s"])

    def backward(self, dout, stream=None):
        if self._inputs is None:
            raise RuntimeError("backward() needs a forward() first")
        x, W_r, W_up, W_gate, W_down, bias = self._inputs
        g = self.grads()
        moe_backward(self.cfg, x, W_r, W_up, W_gate, W_down, self.logits, self.topk_idx, self.gate,
                     self.slot_of, self.perm_token, self.offsets, self.x_perm, self.h_saved,
                     self.act, self.y_perm, self.stats, dout, g["dx"], g["dW_r"],
                     g["dbias"] if bias is not None else None, g["dW_up"], g["dW_gate"],
                     g["dW_down"], self.ws, stream, shared=self.shared_block())
        return g
