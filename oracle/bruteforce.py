"""Brute-force restatement of the MoE forward -- TEST INFRASTRUCTURE ONLY.

Independent of ``moe_oracle.c``: written in the per-expert boolean-mask form
("for each expert, take the tokens routed to it, run the expert, scatter the
weighted result back") of the "Twinkle adapts DeepSeek-V4 training" notes,
§3.2 (MoEBlock.forward), with numpy whole-array ops.  Used on tiny inputs to
pin the C oracle; never fast, never used by the GPU path.
"""
from __future__ import annotations

import math

import numpy as np


def _silu(z):
    return z / (1.0 + np.exp(-z))


def capacity(T, k, E, capacity_factor):
    if not capacity_factor > 0:
        return T
    return min(T, int(math.ceil(float(capacity_factor) * T * k / E)))


def topk_by_sort(logits, k):
    """Full stable sort per token: key (logit descending, NaN last, id ascending)."""
    T, E = logits.shape
    out = np.empty((T, k), np.int32)
    for t in range(T):
        row = logits[t]
        key = np.where(np.isnan(row), -np.inf, row)
        nan_rank = np.isnan(row).astype(np.int64)
        order = np.lexsort((np.arange(E), -key, nan_rank))
        out[t] = order[:k]
    return out


def forward(x, Wr, Wup, Wdown, k, capacity_factor=0.0, Wgate=None, bias=None, noise=None,
            normalize_gates=True, logits=None, temperature=1.0, straight_through=False,
            mask=None, shared=None):
    """Returns (out, topk_idx, gate, kept_mask[T,k]).  Masked tokens (mask 0)
    are routed nowhere: topk -1, gates 0.  ``shared`` = (Wup_s, Wdown_s, Wgate_s
    or None): a dense FFN that every token also passes through, weight 1."""
    x = np.asarray(x, np.float64)
    T, d = x.shape
    E = Wr.shape[1]
    if logits is None:
        logits = x @ np.asarray(Wr, np.float64)
        if bias is not None:
            logits = logits + np.asarray(bias, np.float64)[None, :]
        if noise is not None and not straight_through:
            logits = logits + np.asarray(noise, np.float64)
    logits = np.asarray(logits, np.float64)
    z = logits / temperature
    probs = np.exp(z - z.max(axis=1, keepdims=True))
    probs /= probs.sum(axis=1, keepdims=True)
    key = logits
    if straight_through and noise is not None:
        key = (logits.astype(np.float32) + np.asarray(noise, np.float32)).astype(np.float64)
    topk = topk_by_sort(key, k)
    sel = np.take_along_axis(z, topk, axis=1)
    if straight_through:
        gate = np.ones((T, k))
    elif normalize_gates:
        w = np.exp(sel - sel.max(axis=1, keepdims=True))
        gate = w / w.sum(axis=1, keepdims=True)
    else:
        gate = np.take_along_axis(probs, topk, axis=1)
    if mask is not None:
        pad = np.asarray(mask) == 0
        topk[pad] = -1
        gate[pad] = 0.0

    # routing matrix [T, E] of slot indices (-1 = not selected), then capacity
    C = capacity(T, k, E, capacity_factor)
    kept = np.zeros((T, k), bool)
    for e in range(E):
        tok, slot = np.nonzero(topk == e)          # row-major => ascending token order (masked: -1)
        keep = np.arange(len(tok)) < C
        kept[tok[keep], slot[keep]] = True

    out = np.zeros((T, d))
    for e in range(E):
        sel_e = (topk == e) & kept                   # [T, k]
        tok, slot = np.nonzero(sel_e)
        if len(tok) == 0:
            continue
        xe = x[tok]
        if Wgate is None:
            a = _silu(xe @ np.asarray(Wup[e], np.float64))
        else:
            a = _silu(xe @ np.asarray(Wgate[e], np.float64)) * (xe @ np.asarray(Wup[e], np.float64))
        ye = a @ np.asarray(Wdown[e], np.float64)
        np.add.at(out, tok, gate[tok, slot][:, None] * ye)
    if shared is not None:
        Wus, Wds, Wgs = (None if a is None else np.asarray(a, np.float64) for a in shared)
        a = _silu(x @ Wus) if Wgs is None else _silu(x @ Wgs) * (x @ Wus)
        out = out + a @ Wds
    return out, topk, gate, kept
