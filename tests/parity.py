"""Helpers for GPU-vs-oracle parity tests (imported by tests and the smoke check).

The CUDA path runs through the C ABI (the ctypes binding); the oracle runs on
the same seeded inputs in fp64.  Comparisons:
  * routing indices, counts, offsets, permutation: bit-exact, with the oracle's
    route stage fed the GPU's fp32 logits (the same values decide the top-k);
  * floating-point tensors: relative Frobenius error within the tolerance of
    the layer dtype (1e-5 fp32, 2e-2 bf16);
  * independent routing (oracle logits in fp64): identical top-k except on
    tokens whose k-th / (k+1)-th logit gap is below 1e-4, which are counted.
"""
from __future__ import annotations

import numpy as np
import torch

import moe_inputs
import oracle
import top_routing_expert_moe_gb300 as moe

TOL = {"fp32": 1e-5, "bf16": 2e-2}
NEAR_TIE = 1e-4


def rel_fro(got, want) -> float:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    den = float(np.linalg.norm(want))
    num = float(np.linalg.norm(got - want))
    return num / den if den > 0 else num


to_torch = moe.tensor_from_numpy
gpu_cfg = moe.config_for


def np64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def row_rel(got, want, floor_frac=1e-3) -> np.ndarray:
    """Per-row relative error ||got_i - want_i|| / max(||want_i||, floor), the
    floor being floor_frac times the RMS row norm (rows that are zero or tiny in
    the reference are measured against a typical row instead)."""
    want = np.asarray(want, np.float64)
    if want.size == 0:
        return np.zeros(0)
    got = np.asarray(got, np.float64).reshape(len(want), -1)
    want = want.reshape(len(want), -1)
    wn = np.linalg.norm(want, axis=1)
    floor = floor_frac * float(np.sqrt(np.mean(wn * wn))) + 1e-300
    return np.linalg.norm(got - want, axis=1) / np.maximum(wn, floor)


# Per-row bound beside the whole-tensor Frobenius tolerance: one row that is
# wrong (dropped, zeroed, another token's) has relative error near 1 however
# many correct rows surround it, while rounding leaves every row within a small
# multiple of the tolerance (bf16: a few 2^-9 roundings of intermediates and
# outputs per element, about 4e-3 per row; fp32: about 1e-6).
ROW_TOL = {"fp32": 1e-4, "bf16": 5e-2}


def check_rows(report, key, got, want, dtype):
    """Record the worst row's relative error as report[key] and assert ROW_TOL."""
    rr = row_rel(got, want)
    worst = float(rr.max()) if rr.size else 0.0
    report[key] = worst
    assert worst <= ROW_TOL[dtype], (key, worst, int(rr.argmax()) if rr.size else -1)


def oracle_cfg(w: moe_inputs.Workload, pad_m=128, normalize=True, temperature=1.0,
               straight_through=False) -> oracle.OracleConfig:
    return oracle.OracleConfig(T=w.T, d=w.d, f=w.f, E=w.E, k=w.k,
                               capacity_factor=float(np.float32(w.capacity_factor)),
                               swiglu=w.swiglu, normalize_gates=normalize,
                               aux_coef=float(np.float32(w.aux_coef)), pad_m=pad_m,
                               temperature=float(np.float32(temperature)),
                               straight_through=bool(straight_through), f_shared=w.f_shared)


def f64_inputs(w, inp):
    return {k: (v if k == "mask" else
                moe_inputs.as_f64(v, w.dtype if k not in ("bias", "noise") else "fp32"))
            for k, v in inp.items()}


def run_gpu(w, inp, pad_m=128, normalize=True, backward=True, temperature=1.0,
            straight_through=False):
    """Forward (and the backward sub-steps with their intermediates) on the GPU.
    ``inp["mask"]`` (uint8 [T], 0 = padding token) is optional."""
    cfg = gpu_cfg(w, pad_m, normalize, temperature, straight_through)
    dt = w.dtype
    x = to_torch(inp["x"], dt)
    Wr = to_torch(inp["W_r"], dt)
    Wu = to_torch(inp["W_up"], dt)
    Wg = to_torch(inp.get("W_gate"), dt)
    Wd = to_torch(inp["W_down"], dt)
    b = to_torch(inp.get("bias"), "fp32")
    nz = to_torch(inp.get("noise"), "fp32")
    mk = to_torch(inp.get("mask"), "u8")
    shared = None
    if w.f_shared > 0:
        shared = (to_torch(inp["W_up_s"], dt), to_torch(inp["W_down_s"], dt),
                  to_torch(inp.get("W_gate_s"), dt))
    L = moe.MoELayer(cfg)
    L.forward(x, Wr, Wu, Wd, W_gate=Wg, bias=b, noise=nz, token_mask=mk, shared=shared)
    res = dict(cfg=cfg, layer=L)
    if backward:
        dout = to_torch(inp["dout"], dt)
        R, dev, tdt = L.rows_cap, x.device, cfg.torch_dtype
        dy = torch.empty(R, w.d, dtype=tdt, device=dev)
        dgate = torch.empty(w.T, w.k, dtype=torch.float32, device=dev)
        dh = torch.empty(cfg.nh, R, w.f, dtype=tdt, device=dev)
        dxp = torch.empty(R, w.d, dtype=tdt, device=dev)
        dlogits = torch.empty(w.T, w.E, dtype=torch.float32, device=dev)
        g = L.grads()
        sh = None
        if w.f_shared > 0:
            Ts = L.shared_rows
            res["dh_shared"] = torch.empty(cfg.nh, Ts, w.f_shared, dtype=tdt, device=dev)
            res["dx_shared"] = torch.empty(Ts, w.d, dtype=tdt, device=dev)
            sh = L.shared_block(dout=dout, dh=res["dh_shared"], dx=res["dx_shared"])
        moe.moe_combine_backward(cfg, dout, L.y_perm, L.gate, L.slot_of, L.perm_token, L.offsets,
                                 dy, dgate)
        moe.moe_grouped_ffn_backward(cfg, L.x_perm, L.offsets, Wu, Wg, Wd, L.h_saved, L.act, dy,
                                     dh, dxp, g["dW_up"], g["dW_gate"], g["dW_down"], L.ws,
                                     shared=sh)
        moe.moe_router_backward(cfg, x, Wr, L.logits, L.topk_idx, L.gate, L.slot_of, dgate, dxp,
                                L.stats, g["dx"], g["dW_r"], g["dbias"] if b is not None else None,
                                dlogits, L.ws, shared=sh)
        res.update(dy=dy, dgate=dgate, dh=dh, dxp=dxp, dlogits=dlogits, grads=g, dout=dout)
    torch.cuda.synchronize()
    res["status"] = moe.last_device_status()
    return res


def check_routing(w, ocfg, r, inp64, report):
    """Route/permute parity.  Returns the conditioned oracle forward."""
    L = r["layer"]
    logits = np64(L.logits)
    noise, mask = inp64.get("noise"), inp64.get("mask")
    st_mode = ocfg.straight_through
    # logits vs fp64 oracle (straight-through: the noise enters only the selection)
    ol = oracle.router_logits(ocfg, inp64["x"], inp64["W_r"], inp64.get("bias"),
                              None if st_mode else noise)
    report["logits_rel"] = rel_fro(logits, ol)
    # conditioned oracle: route the GPU's fp32 logits
    o = oracle.forward(ocfg, inp64["x"], inp64["W_r"], inp64["W_up"], inp64["W_down"],
                       Wgate=inp64.get("W_gate"), noise=noise, logits_in=logits, mask=mask,
                       Wup_s=inp64.get("W_up_s"), Wdown_s=inp64.get("W_down_s"),
                       Wgate_s=inp64.get("W_gate_s"))
    topk = L.topk_idx.cpu().numpy()
    assert (topk == o["topk_idx"]).all(), "top-k differs from the oracle on the same logits"
    assert (L.counts.cpu().numpy() == o["counts"]).all(), "counts differ"
    assert (L.kept.cpu().numpy() == o["kept"]).all(), "kept differs"
    assert (L.offsets.cpu().numpy() == o["offsets"]).all(), "offsets differ"
    rows = int(o["offsets"][-1])
    assert (L.perm_token.cpu().numpy()[:rows] == o["perm_token"]).all(), "perm_token differs"
    assert (L.slot_of.cpu().numpy() == o["slot_of"]).all(), "slot_of differs"
    report["gate_rel"] = rel_fro(np64(L.gate), o["gate"])
    st = np64(L.stats)
    report["pbar_rel"] = rel_fro(st[moe.STAT_PBAR:], o["stats"][oracle.ST_PBAR:])
    report["aux_loss"] = (float(st[moe.STAT_AUX_LOSS]), float(o["stats"][oracle.ST_AUX_LOSS]))
    for i in (moe.STAT_AUX_SWITCH, moe.STAT_ENTROPY):
        assert abs(st[i] - o["stats"][i]) <= 1e-4 * max(1.0, abs(o["stats"][i])), (i, st[i], o["stats"][i])
    assert abs(st[moe.STAT_AUX_LOSS] - o["stats"][oracle.ST_AUX_LOSS]) <= \
        1e-3 * abs(o["stats"][oracle.ST_AUX_LOSS]) + 1e-9
    for i in (moe.STAT_NONFINITE, moe.STAT_DROPPED, moe.STAT_TOKENS):
        assert st[i] == o["stats"][i], (i, st[i], o["stats"][i])
    for i in (moe.STAT_MAX_OVER_MEAN_KEPT, moe.STAT_COUNT_CV, moe.STAT_MAX_OVER_MEAN_COUNT):
        assert abs(st[i] - o["stats"][i]) <= 1e-5 * max(1.0, abs(o["stats"][i])), (i, st[i], o["stats"][i])
    # independent routing (oracle's own fp64 logits)
    oi = oracle.route(ocfg, ol, noise if st_mode else None, mask)
    key = (ol.astype(np.float32) + noise.astype(np.float32)).astype(np.float64) \
        if st_mode and noise is not None else ol
    srt = -np.sort(-key, axis=1)
    gap = srt[:, ocfg.k - 1] - srt[:, ocfg.k] if ocfg.k < ocfg.E else np.full(ocfg.T, np.inf)
    near = gap < NEAR_TIE
    same = (np.sort(oi["topk_idx"], 1) == np.sort(topk, 1)).all(1)
    report["near_tie_tokens"] = int(near.sum())
    report["independent_mismatch_excluded"] = int((~same & near).sum())
    assert same[~near].all(), f"independent routing differs on {int((~same & ~near).sum())} clear tokens"
    return o


def rows_of(t, idx) -> np.ndarray:
    """fp64 copy of rows idx of a device tensor (only those rows leave the GPU,
    so uninitialised rows past the layout's end are never converted)."""
    idx = np.asarray(idx, np.int64)
    if idx.size == 0:
        return np.zeros((0,) + tuple(t.shape[1:]))
    return np64(t[torch.as_tensor(idx, device=t.device, dtype=torch.long)])


def check_forward(w, ocfg, r, o, inp64, report, sample_rows=None):
    L = r["layer"]
    tol = TOL[w.dtype]
    rows = int(o["offsets"][-1])
    # x_perm rows are exact copies; padding rows zero
    xp = np64(L.x_perm[:rows])
    perm = o["perm_token"]
    real = perm >= 0
    assert np.array_equal(xp[real], inp64["x"][perm[real]]), "x_perm rows differ"
    assert (xp[~real] == 0).all(), "padding rows of x_perm are not zero"
    # per-row expert stage (sampled)
    idx = np.nonzero(real)[0]
    if sample_rows is not None and len(idx) > sample_rows:
        idx = np.sort(np.random.default_rng(0).choice(idx, sample_rows, replace=False))
    row_e = np.searchsorted(o["offsets"], idx, side="right") - 1
    want_h, want_u, want_a, want_y = [], [], [], []
    for rr, e in zip(idx, row_e):
        ef = oracle.expert_forward(ocfg, e, inp64["x"][perm[rr]], inp64["W_up"], inp64["W_down"],
                                   inp64.get("W_gate"))
        want_h.append(ef["h"]); want_a.append(ef["act"]); want_y.append(ef["y"])
        if ocfg.swiglu:
            want_u.append(ef["u"])
    out = np64(L.out)
    report["out_rel"] = rel_fro(out, o["out"])
    check_rows(report, "out_row_max", out, o["out"], w.dtype)
    if ocfg.f_shared > 0:
        check_shared_forward(w, ocfg, L, inp64, report, sample_rows)
    if len(idx) == 0:        # nothing routed (e.g. every token is padding)
        if ocfg.f_shared == 0:
            assert (out == 0).all(), "out is not zero with no routed token"
        assert report["out_rel"] <= tol, ("out_rel", report["out_rel"], tol)
        return
    H0, A, Y = rows_of(L.h_saved[0], idx), rows_of(L.act, idx), rows_of(L.y_perm, idx)
    report["h_rel"] = rel_fro(H0, np.array(want_h))
    check_rows(report, "h_row_max", H0, np.array(want_h), w.dtype)
    if ocfg.swiglu:
        H1 = rows_of(L.h_saved[1], idx)
        report["u_rel"] = rel_fro(H1, np.array(want_u))
        check_rows(report, "u_row_max", H1, np.array(want_u), w.dtype)
    report["act_rel"] = rel_fro(A, np.array(want_a))
    check_rows(report, "act_row_max", A, np.array(want_a), w.dtype)
    report["y_rel"] = rel_fro(Y, np.array(want_y))
    check_rows(report, "y_row_max", Y, np.array(want_y), w.dtype)
    for key in ("h_rel", "u_rel", "act_rel", "y_rel", "out_rel"):
        if key in report:
            assert report[key] <= tol, (key, report[key], tol)


def check_shared_forward(w, ocfg, L, inp64, report, sample_rows=None):
    """Shared experts' h / act / y rows (sampled) against the oracle's FFN; the
    rows past T are zero."""
    T = ocfg.T
    toks = np.arange(T)
    if sample_rows is not None and T > sample_rows:
        toks = np.sort(np.random.default_rng(1).choice(T, sample_rows, replace=False))
    want = [oracle.shared_forward(ocfg, inp64["x"][t], inp64["W_up_s"], inp64["W_down_s"],
                                  inp64.get("W_gate_s")) for t in toks]
    H, A, Y = np64(L.h_shared), np64(L.act_shared), np64(L.y_shared)
    report["h_shared_rel"] = rel_fro(H[0][toks], np.array([q["h"] for q in want]))
    if ocfg.swiglu:
        report["u_shared_rel"] = rel_fro(H[1][toks], np.array([q["u"] for q in want]))
    report["act_shared_rel"] = rel_fro(A[toks], np.array([q["act"] for q in want]))
    report["y_shared_rel"] = rel_fro(Y[toks], np.array([q["y"] for q in want]))
    assert (Y[T:] == 0).all() and (A[T:] == 0).all(), "shared rows past T are not zero"
    tol = TOL[w.dtype]
    for key in ("h_shared_rel", "u_shared_rel", "act_shared_rel", "y_shared_rel"):
        if key in report:
            assert report[key] <= tol, (key, report[key], tol)


def check_backward(w, ocfg, r, o, inp64, report, with_bias):
    L = r["layer"]
    tol = TOL[w.dtype]
    logits = np64(L.logits)
    ob = oracle.backward(ocfg, inp64["x"], inp64["W_r"], inp64["W_up"], inp64["W_down"], logits,
                         o["topk_idx"], o["gate"], o["slot_of"], inp64["dout"],
                         Wgate=inp64.get("W_gate"), with_bias=with_bias, per_slot=True,
                         Wup_s=inp64.get("W_up_s"), Wdown_s=inp64.get("W_down_s"),
                         Wgate_s=inp64.get("W_gate_s"))
    g = r["grads"]
    slot = o["slot_of"]
    kept = slot >= 0
    # dgate and the per-slot intermediates
    report["dgate_rel"] = rel_fro(np64(r["dgate"]), ob["dgate"])
    tt, jj = np.nonzero(kept)
    rows = slot[tt, jj]
    gate = o["gate"]
    dy = rows_of(r["dy"], rows)
    dy_want = gate[tt, jj][:, None] * inp64["dout"][tt]
    report["dy_rel"] = rel_fro(dy, dy_want)
    check_rows(report, "dy_row_max", dy, dy_want, w.dtype)
    pad_rows = np.nonzero(o["perm_token"] < 0)[0]
    assert (rows_of(r["dy"], pad_rows) == 0).all(), "padding rows of dy_perm are not zero"
    dh0 = rows_of(r["dh"][0], rows)
    report["dh_rel"] = rel_fro(dh0, ob["dh_slot"][tt, jj, 0])
    check_rows(report, "dh_row_max", dh0, ob["dh_slot"][tt, jj, 0], w.dtype)
    if ocfg.swiglu:
        dh1 = rows_of(r["dh"][1], rows)
        report["du_rel"] = rel_fro(dh1, ob["dh_slot"][tt, jj, 1])
        check_rows(report, "du_row_max", dh1, ob["dh_slot"][tt, jj, 1], w.dtype)
    dxp = rows_of(r["dxp"], rows)
    report["dxp_rel"] = rel_fro(dxp, ob["dxp_slot"][tt, jj])
    check_rows(report, "dxp_row_max", dxp, ob["dxp_slot"][tt, jj], w.dtype)
    report["dlogits_rel"] = rel_fro(np64(r["dlogits"]), ob["dlogits"])
    dx = np64(g["dx"])
    report["dx_rel"] = rel_fro(dx, ob["dx"])
    check_rows(report, "dx_row_max", dx, ob["dx"], w.dtype)
    report["dWr_rel"] = rel_fro(np64(g["dW_r"]), ob["dWr"])
    report["dWup_rel"] = rel_fro(np64(g["dW_up"]), ob["dWup"])
    report["dWdown_rel"] = rel_fro(np64(g["dW_down"]), ob["dWdown"])
    if ocfg.swiglu:
        report["dWgate_rel"] = rel_fro(np64(g["dW_gate"]), ob["dWgate"])
    if with_bias:
        report["db_rel"] = rel_fro(np64(g["dbias"]), ob["db"])
    if ocfg.f_shared > 0:
        report["dWup_s_rel"] = rel_fro(np64(g["dW_up_s"]), ob["dWup_s"])
        report["dWdown_s_rel"] = rel_fro(np64(g["dW_down_s"]), ob["dWdown_s"])
        if ocfg.swiglu:
            report["dWgate_s_rel"] = rel_fro(np64(g["dW_gate_s"]), ob["dWgate_s"])
    for key, v in list(report.items()):
        if key.startswith("d") and key.endswith("_rel"):
            assert v <= tol, (key, v, tol)


def full_check(w, inp, pad_m=128, normalize=True, backward=True, sample_rows=None,
               temperature=1.0, straight_through=False):
    report = {}
    r = run_gpu(w, inp, pad_m=pad_m, normalize=normalize, backward=backward,
                temperature=temperature, straight_through=straight_through)
    assert r["status"] == 0, f"device status {r['status']}"
    ocfg = oracle_cfg(w, pad_m, normalize, temperature, straight_through)
    inp64 = f64_inputs(w, inp)
    o = check_routing(w, ocfg, r, inp64, report)
    check_forward(w, ocfg, r, o, inp64, report, sample_rows=sample_rows)
    if backward:
        check_backward(w, ocfg, r, o, inp64, report, with_bias=inp.get("bias") is not None)
    return report, r
