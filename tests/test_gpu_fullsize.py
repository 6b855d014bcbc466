"""GPU parity at the full workload sizes the benchmark times.

The whole layer runs at full size through the C ABI (the same calls and
buffers bench.py uses).  Then:
  * routing, counts, capacity drops and the permutation are compared bit-exact
    on every token, with the oracle's route stage fed the GPU's fp32 logits;
  * per-token quantities (logits, output, dgate, dh and dx_perm of each kept
    slot, dlogits, dx) are compared with the oracle on a seeded token sample
    (the aux term of the sample's backward uses the full batch's pbar and T);
  * the weight-gradient reductions, which no per-token oracle call can give at
    this size, are checked entry-wise as fp64 sums over the GPU's own operands
    (x_perm, act, dy, dh, dlogits), operands the sample checks above validate.
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
    rep["out_rel"] = parity.rel_fro(_rows(L.out, S), out_want)
    ob = oracle.backward(sub, xs, Wr, Wu, Wd, logits[S], ro["topk_idx"][S], ro["gate"][S],
                         slot[S], f64(inp["dout"][S]), Wgate=Wg, per_slot=True,
                         pbar=st[oracle.ST_PBAR:], T_aux=T, with_bias=b is not None)
    rep["dgate_rel"] = parity.rel_fro(_rows(r["dgate"], S), ob["dgate"])
    rep["dlogits_rel"] = parity.rel_fro(_rows(r["dlogits"], S), ob["dlogits"])
    rep["dx_rel"] = parity.rel_fro(_rows(g["dx"], S), ob["dx"])
    ii, jj = np.nonzero(slot[S] >= 0)
    srow = slot[S][ii, jj]
    rep["dxp_rel"] = parity.rel_fro(_rows(r["dxp"], srow), ob["dxp_slot"][ii, jj])
    dh = r["dh"]
    rep["dh_rel"] = parity.rel_fro(_rows(dh[0], srow), ob["dh_slot"][ii, jj, 0])
    if w.swiglu:
        rep["du_rel"] = parity.rel_fro(_rows(dh[1], srow), ob["dh_slot"][ii, jj, 1])
    # ---- reductions: sampled entries as fp64 sums over the GPU operands
    off = po["offsets"]
    kept = po["kept"]

    def seg_sum(A, B, e, a_col, b_col):
        lo, hi = int(off[e]), int(off[e] + kept[e])
        if hi == lo:
            return 0.0
        a = parity.np64(A[lo:hi, a_col])
        bb = parity.np64(B[lo:hi, b_col])
        return float(a @ bb)

    ents = [(int(rng.integers(E)), int(rng.integers(w.f)), int(rng.integers(w.d)))
            for _ in range(n_entries)]
    got = np.array([float(g["dW_down"][e, j, i]) for e, j, i in ents])
    want = np.array([seg_sum(L.act, r["dy"], e, j, i) for e, j, i in ents])
    rep["dWdown_rel"] = parity.rel_fro(got, want)
    dh_up = dh[1] if w.swiglu else dh[0]
    got = np.array([float(g["dW_up"][e, i, j]) for e, j, i in ents])
    want = np.array([seg_sum(L.x_perm, dh_up, e, i, j) for e, j, i in ents])
    rep["dWup_rel"] = parity.rel_fro(got, want)
    if w.swiglu:
        got = np.array([float(g["dW_gate"][e, i, j]) for e, j, i in ents])
        want = np.array([seg_sum(L.x_perm, dh[0], e, i, j) for e, j, i in ents])
        rep["dWgate_rel"] = parity.rel_fro(got, want)
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
