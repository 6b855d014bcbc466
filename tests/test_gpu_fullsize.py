"""GPU parity at the full workload sizes the benchmark times.

The whole layer runs at full size through the C ABI (the same calls and
buffers bench.py uses).  Then:
  * routing, counts, capacity drops and the permutation are compared bit-exact
    on every token, with the oracle's route stage fed the GPU's fp32 logits;
  * per-token quantities (logits, output, dgate, dh and dx_perm of each kept
    slot, dlogits, dx) are compared with the oracle on a seeded token sample
    (the aux term of the sample's backward uses the full batch's pbar and T);
  * sampled rows also meet a per-row relative bound (parity.ROW_TOL), so one
    wrong row cannot hide inside a whole-tensor norm;
  * sampled entries of dW_down / dW_up / dW_gate come from the oracle's
    per-entry definition over the expert's kept tokens of the whole batch
    (variable-length reductions of up to ~16k rows); dW_r entries are fp64
    sums of x against the GPU's dlogits, whose rows the sample checks.
"""
import numpy as np
import pytest
import torch

import moe_inputs
import oracle
import top_routing_expert_moe_gb300 as moe
from tests import parity

pytestmark = pytest.mark.gpu


def _rows(t, idx):
    return parity.np64(t[torch.as_tensor(idx, device=t.device, dtype=torch.long)])


def fullsize_check(w, inp, n_tok, n_entries=48, seed=0):
    tol = parity.TOL[w.dtype]
    rep = {}
    r = parity.run_gpu(w, inp)
    assert r["status"] == 0
    L, g = r["layer"], r["grads"]
    ocfg = parity.oracle_cfg(w)
    T, E, k = w.T, w.E, w.k
    # ---- routing on every token (bit-exact)
    logits = parity.np64(L.logits)
    ro = oracle.route(ocfg, logits)
    assert (L.topk_idx.cpu().numpy() == ro["topk_idx"]).all()
    assert (L.counts.cpu().numpy() == ro["counts"]).all()
    po = oracle.permute(ocfg, ro["topk_idx"])
    assert (L.kept.cpu().numpy() == po["kept"]).all()
    assert (L.offsets.cpu().numpy() == po["offsets"]).all()
    rows = int(po["offsets"][-1])
    assert (L.perm_token[:rows].cpu().numpy() == po["perm_token"]).all()
    slot = L.slot_of.cpu().numpy()
    assert (slot == po["slot_of"]).all()
    rep["gate_rel"] = parity.rel_fro(parity.np64(L.gate), ro["gate"])
    st = oracle.stats(ocfg, ro["probs"], ro["topk_idx"], ro["counts"], po["kept"], ro["nonfinite"])
    gst = parity.np64(L.stats)
    rep["pbar_rel"] = parity.rel_fro(gst[moe.STAT_PBAR:], st[oracle.ST_PBAR:])
    assert gst[moe.STAT_DROPPED] == st[oracle.ST_DROPPED]
    rep["dropped"] = int(st[oracle.ST_DROPPED])
    # ---- per-token sample against the oracle
    rng = np.random.default_rng(seed)
    S = np.sort(rng.choice(T, n_tok, replace=False))
    dropped_tok = np.nonzero((slot < 0).any(1))[0]
    if len(dropped_tok):                       # include tokens that lost a slot
        S = np.unique(np.concatenate([S, dropped_tok[:2]]))
    f64 = lambda a, dt=w.dtype: moe_inputs.as_f64(a, dt)  # noqa: E731
    xs = f64(inp["x"][S])
    Wr, Wu, Wd = f64(inp["W_r"]), f64(inp["W_up"]), f64(inp["W_down"])
    Wg = f64(inp["W_gate"]) if inp["W_gate"] is not None else None
    sub = parity.oracle_cfg(w)
    sub.T = len(S)
    b = inp["bias"].astype(np.float64) if inp["bias"] is not None else None
    nz = inp["noise"][S].astype(np.float64) if inp["noise"] is not None else None
    rep["logits_rel"] = parity.rel_fro(logits[S], oracle.router_logits(sub, xs, Wr, b, nz))
    out_want = np.zeros((len(S), w.d))
    for i, t in enumerate(S):
        for j in range(k):
            if slot[t, j] >= 0:
                y = oracle.expert_apply(ocfg, ro["topk_idx"][t, j], xs[i], Wu, Wg, Wd)
                out_want[i] += ro["gate"][t, j] * y
    out_got = _rows(L.out, S)
    rep["out_rel"] = parity.rel_fro(out_got, out_want)
    parity.check_rows(rep, "out_row_max", out_got, out_want, w.dtype)
    ob = oracle.backward(sub, xs, Wr, Wu, Wd, logits[S], ro["topk_idx"][S], ro["gate"][S],
                         slot[S], f64(inp["dout"][S]), Wgate=Wg, per_slot=True,
                         pbar=st[oracle.ST_PBAR:], T_aux=T, with_bias=b is not None)
    rep["dgate_rel"] = parity.rel_fro(_rows(r["dgate"], S), ob["dgate"])
    rep["dlogits_rel"] = parity.rel_fro(_rows(r["dlogits"], S), ob["dlogits"])
    dx_got = _rows(g["dx"], S)
    rep["dx_rel"] = parity.rel_fro(dx_got, ob["dx"])
    parity.check_rows(rep, "dx_row_max", dx_got, ob["dx"], w.dtype)
    ii, jj = np.nonzero(slot[S] >= 0)
    srow = slot[S][ii, jj]
    dxp_got = _rows(r["dxp"], srow)
    rep["dxp_rel"] = parity.rel_fro(dxp_got, ob["dxp_slot"][ii, jj])
    parity.check_rows(rep, "dxp_row_max", dxp_got, ob["dxp_slot"][ii, jj], w.dtype)
    dh = r["dh"]
    dh_got = _rows(dh[0], srow)
    rep["dh_rel"] = parity.rel_fro(dh_got, ob["dh_slot"][ii, jj, 0])
    parity.check_rows(rep, "dh_row_max", dh_got, ob["dh_slot"][ii, jj, 0], w.dtype)
    if w.swiglu:
        du_got = _rows(dh[1], srow)
        rep["du_rel"] = parity.rel_fro(du_got, ob["dh_slot"][ii, jj, 1])
        parity.check_rows(rep, "du_row_max", du_got, ob["dh_slot"][ii, jj, 1], w.dtype)
    # ---- expert weight gradients: sampled entries from the oracle's per-entry
    # definition over each sampled expert's kept tokens (the whole batch)
    off, kept = po["offsets"], po["kept"]
    perm = po["perm_token"]
    busy = np.nonzero(kept > 0)[0]
    kinds = [(oracle.WGRAD_DOWN, "dW_down", w.f, w.d), (oracle.WGRAD_UP, "dW_up", w.d, w.f)]
    if w.swiglu:
        kinds.append((oracle.WGRAD_GATE, "dW_gate", w.d, w.f))
    got_all = {name: [] for _, name, _, _ in kinds}
    want_all = {name: [] for _, name, _, _ in kinds}
    for e in rng.choice(busy, size=min(3, len(busy)), replace=False):
        e = int(e)
        r0_, n_e = int(off[e]), int(kept[e])
        toks = perm[r0_:r0_ + n_e]
        assert (np.diff(toks) > 0).all()
        jsel = np.argmax(slot[toks] == (r0_ + np.arange(n_e))[:, None], axis=1)
        gates = ro["gate"][toks, jsel]
        Wg_e = f64(inp["W_gate"][e]) if w.swiglu else None
        xs_e, do_e = f64(inp["x"][toks]), f64(inp["dout"][toks])
        Wu_e, Wd_e = f64(inp["W_up"][e]), f64(inp["W_down"][e])
        for kind, name, nr, nc in kinds:
            rr = rng.integers(nr, size=n_entries // 3)
            cc = rng.integers(nc, size=n_entries // 3)
            want_all[name].append(oracle.expert_wgrad_entries(
                ocfg, xs_e, gates, do_e, Wu_e, Wd_e, np.full(len(rr), kind), rr, cc, Wg_e=Wg_e))
            gt = g[name][e]
            got_all[name].append(parity.np64(gt[torch.as_tensor(rr, device=gt.device),
                                                torch.as_tensor(cc, device=gt.device)]))
        del xs_e, do_e, Wu_e, Wd_e, Wg_e
    for _, name, _, _ in kinds:
        key = {"dW_down": "dWdown_rel", "dW_up": "dWup_rel", "dW_gate": "dWgate_rel"}[name]
        rep[key] = parity.rel_fro(np.concatenate(got_all[name]), np.concatenate(want_all[name]))
    x_gpu = parity.to_torch(inp["x"], w.dtype)
    dl = r["dlogits"]
    cols = rng.integers(w.d, size=16)
    got = np.array([[float(g["dW_r"][i, e]) for e in range(E)] for i in cols])
    want = np.array([[float(parity.np64(x_gpu[:, i]) @ parity.np64(dl[:, e])) for e in range(E)]
                     for i in cols])
    rep["dWr_rel"] = parity.rel_fro(got, want)
    if b is not None:
        rep["db_rel"] = parity.rel_fro(parity.np64(g["dbias"]), parity.np64(dl.sum(0)))
    print(f"\n[{w.name} full size] " + str({k_: (round(v, 6) if isinstance(v, float) else v)
                                             for k_, v in rep.items()}))
    for key, v in rep.items():
        if key.endswith("_rel"):
            assert v <= tol, (key, v)
    return rep


def test_llama4_shape_full_size():
    w = moe_inputs.get("llama4_bf16")
    fullsize_check(w, moe_inputs.make_inputs(w, 0), n_tok=16)


def test_skewed16_shape_full_size():
    w = moe_inputs.get("skewed16_bf16")
    rep = fullsize_check(w, moe_inputs.make_inputs(w, 0), n_tok=16)
    assert rep["dropped"] > 0


@pytest.mark.parametrize("T", moe_inputs.MIXTRAL_SWEEP_T)
def test_mixtral_shape_full_size(T):
    w = moe_inputs.get("mixtral_bf16").with_tokens(T)
    fullsize_check(w, moe_inputs.make_inputs(w, 0), n_tok=6)
