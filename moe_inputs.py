"""Seeded synthetic workloads for the sparse MoE layer.

This module holds the workload shapes and the seeded input generators that
both the CUDA path (tests, bench) and the CPU oracle consume.  It contains
none of the layer's arithmetic: only random draws, bf16 rounding of the draws
and the stored router-bias recipe of the skewed-routing workload.

Each tensor has its own PCG64 stream keyed by (seed, tensor id), so a tensor
does not depend on which others are drawn.  bf16 tensors are fp32 normals
rounded to nearest-even and kept as their uint16 bit patterns; ``as_f64``
gives the exact values the oracle uses.
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
ZIPF_BIAS_FILE = os.path.join(_HERE, "tests", "golden", "skewed16_zipf_bias.json")

# fixed stream ids (one per tensor)
_TENSOR_IDS = {"x": 1, "W_r": 2, "bias": 3, "W_up": 4, "W_gate": 5, "W_down": 6,
               "noise": 7, "dout": 8, "gumbel": 9, "mask": 10, "W_up_s": 11, "W_gate_s": 12,
               "W_down_s": 13}


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    f: int
    E: int
    k: int
    capacity_factor: float      # 0 : no capacity limit
    dtype: str                  # "fp32" or "bf16"
    swiglu: bool = False
    noise_std: float = 0.0      # gate noise N(0, noise_std) added to the logits
    zipf_bias: bool = False     # router bias giving a Zipf(1.1) expert preference
    aux_coef: float = 0.01
    w_std: float = 0.02
    backward: bool = True
    f_shared: int = 0           # hidden width of the shared experts' FFN (0: none)

    def with_tokens(self, T: int) -> "Workload":
        return replace(self, T=T, name=f"{self.name.split('@')[0]}@T{T}")


# The five layer shapes (the last one is swept over T = 4k, 16k, 64k).
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 256, 128, 256, 4, 2, 0.0, "fp32", backward=False),
    "small_bf16": Workload("small_bf16", 2048, 1024, 2048, 4, 2, 1.2, "bf16"),
    "llama4_bf16": Workload("llama4_bf16", 16384, 2048, 4096, 8, 2, 1.2, "bf16", noise_std=0.1),
    "skewed16_bf16": Workload("skewed16_bf16", 65536, 4096, 2816, 16, 2, 1.2, "bf16",
                              zipf_bias=True),
    "mixtral_bf16": Workload("mixtral_bf16", 65536, 4096, 14336, 8, 2, 0.0, "bf16", swiglu=True),
}
MIXTRAL_SWEEP_T = (4096, 16384, 65536)


def get(name: str) -> Workload:
    if "@T" in name:
        base, t = name.split("@T")
        return WORKLOADS[base].with_tokens(int(t))
    return WORKLOADS[name]


# ---------------------------------------------------------------------------
def _rng(seed: int, tensor: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, _TENSOR_IDS[tensor]]))


def bf16_bits(a32: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); return the uint16 bit patterns."""
    u = np.ascontiguousarray(a32, np.float32).view(np.uint32)
    r = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal(seed: int, tensor: str, shape, std: float, dtype: str, chunk: int = 1 << 24):
    """N(0, std) draws of the given shape; bf16 -> uint16 bits, fp32 -> float32."""
    n = int(np.prod(shape))
    g = _rng(seed, tensor)
    out = np.empty(n, np.uint16 if dtype == "bf16" else np.float32)
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        v = g.standard_normal(m, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        out[s:s + m] = bf16_bits(v) if dtype == "bf16" else v
    return out.reshape(shape)


def as_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of a generated tensor."""
    if a is None:
        return None
    if dtype == "bf16" and a.dtype == np.uint16:
        return bf16_to_f32(a).astype(np.float64)
    return np.asarray(a, np.float64)


def zipf_bias(E: int, alpha: float, s: float = 1.1) -> np.ndarray:
    """b_e = alpha * ln(z_e), z the Zipf(s) distribution over expert ranks 1..E."""
    z = 1.0 / np.arange(1, E + 1, dtype=np.float64) ** s
    z /= z.sum()
    return (alpha * np.log(z)).astype(np.float32)


def stored_zipf_alpha() -> float:
    with open(ZIPF_BIAS_FILE) as fh:
        return float(json.load(fh)["alpha"])


def make_inputs(w: Workload, seed: int = 0, parts=("x", "W_r", "bias", "W_up", "W_gate",
                                                    "W_down", "noise", "dout", "shared"),
                zipf_alpha: float | None = None) -> dict:
    """Seeded inputs of workload ``w``.  Router bias and noise are fp32; the rest
    follow ``w.dtype``.  Absent optional tensors are None.  With ``w.f_shared``
    the shared experts' weights W_up_s, W_gate_s (SwiGLU) [d, f_shared] and
    W_down_s [f_shared, d] are drawn too."""
    dt = w.dtype
    out = {}
    if "x" in parts:
        out["x"] = normal(seed, "x", (w.T, w.d), 1.0, dt)
    if "W_r" in parts:
        out["W_r"] = normal(seed, "W_r", (w.d, w.E), w.w_std, dt)
    if "bias" in parts:
        if w.zipf_bias:
            a = stored_zipf_alpha() if zipf_alpha is None else zipf_alpha
            out["bias"] = zipf_bias(w.E, a)
        else:
            out["bias"] = None
    if "W_up" in parts:
        out["W_up"] = normal(seed, "W_up", (w.E, w.d, w.f), w.w_std, dt)
    if "W_gate" in parts:
        out["W_gate"] = normal(seed, "W_gate", (w.E, w.d, w.f), w.w_std, dt) if w.swiglu else None
    if "W_down" in parts:
        out["W_down"] = normal(seed, "W_down", (w.E, w.f, w.d), w.w_std, dt)
    if "noise" in parts:
        out["noise"] = (normal(seed, "noise", (w.T, w.E), w.noise_std, "fp32")
                        if w.noise_std > 0 else None)
    if "dout" in parts:
        out["dout"] = normal(seed, "dout", (w.T, w.d), 1.0, dt)
    if "shared" in parts and w.f_shared > 0:
        fs = w.f_shared
        out["W_up_s"] = normal(seed, "W_up_s", (w.d, fs), w.w_std, dt)
        out["W_gate_s"] = normal(seed, "W_gate_s", (w.d, fs), w.w_std, dt) if w.swiglu else None
        out["W_down_s"] = normal(seed, "W_down_s", (fs, w.d), w.w_std, dt)
    return out


def gumbel(seed: int, T: int, E: int) -> np.ndarray:
    """fp32 [T, E] standard Gumbel draws, -ln(-ln U) with U uniform on (0, 1):
    the selection noise of Gumbel top-k routing."""
    rng = np.random.Generator(np.random.PCG64([seed, _TENSOR_IDS["gumbel"]]))
    u = rng.random((T, E))
    u = np.clip(u, np.finfo(np.float64).tiny, 1.0 - 2.0 ** -53)
    return (-np.log(-np.log(u))).astype(np.float32)


def padding_mask(seed: int, T: int, seq_len: int = 128) -> np.ndarray:
    """uint8 [T] token mask of a right-padded batch (1 = real token, 0 = padding):
    the tokens form sequences of ``seq_len``; each keeps a uniformly drawn real
    length in [seq_len / 2, seq_len], the last sequence is all padding and the
    tokens past the last full sequence are padding too."""
    rng = np.random.Generator(np.random.PCG64([seed, _TENSOR_IDS["mask"]]))
    m = np.zeros(T, np.uint8)
    nseq = T // seq_len
    for s in range(max(nseq - 1, 0)):
        n = int(rng.integers(seq_len // 2, seq_len + 1))
        m[s * seq_len: s * seq_len + n] = 1
    return m
