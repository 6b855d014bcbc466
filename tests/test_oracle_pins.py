"""Pins of the fp64 oracle against things other than itself (CPU only).

* a hand-worked routing example (tests/golden/route_worked_example.json),
* the independent brute-force mask-loop restatement (oracle/bruteforce.py),
* closed forms: one expert = a plain FFN; k = E = a dense softmax mixture;
  a uniform router gives zero variance-form aux loss and Switch form 1,
* structural invariants of the routing,
* central finite differences of <dout, out> + aux loss for every gradient.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import bruteforce

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _frac(s):
    return float(Fraction(s))


def _rand_case(rng, T, d, f, E, k, swiglu=False, bias=False, noise=False, scale=1.0):
    x = rng.standard_normal((T, d))
    Wr = rng.standard_normal((d, E)) * scale
    Wup = rng.standard_normal((E, d, f)) * 0.3
    Wg = rng.standard_normal((E, d, f)) * 0.3 if swiglu else None
    Wd = rng.standard_normal((E, f, d)) * 0.3
    b = rng.standard_normal(E) * 0.5 if bias else None
    nz = rng.standard_normal((T, E)) * 0.1 if noise else None
    return x, Wr, Wup, Wg, Wd, b, nz


# --------------------------------------------------------------------------- golden
def test_worked_example_routing(oracle_lib):
    g = json.load(open(os.path.join(GOLDEN, "route_worked_example.json")))
    c = g["config"]
    cfg = oracle.OracleConfig(T=c["T"], d=1, f=1, E=c["E"], k=c["k"],
                              capacity_factor=c["capacity_factor"], pad_m=c["pad_m"],
                              aux_coef=c["aux_coef"])
    logits = np.log(np.array(g["logit_weights"], np.float64))
    ex = g["expected"]
    r = oracle.route(cfg, logits)
    assert r["topk_idx"].tolist() == ex["topk_idx"]
    assert r["counts"].tolist() == ex["counts"]
    np.testing.assert_allclose(r["gate"], [[_frac(v) for v in row] for row in ex["gate"]], rtol=1e-14)
    np.testing.assert_allclose(r["probs"], [[_frac(v) for v in row] for row in ex["probs"]], rtol=1e-14)
    assert oracle.capacity(cfg) == ex["capacity"]
    p = oracle.permute(cfg, r["topk_idx"])
    assert p["kept"].tolist() == ex["kept"]
    assert p["offsets"].tolist() == ex["offsets"]
    assert p["perm_token"].tolist() == ex["perm_token"]
    assert p["slot_of"].tolist() == ex["slot_of"]
    x = np.zeros((cfg.T, 1))
    W = np.zeros((cfg.E, 1, 1))
    fw = oracle.forward(cfg, x, np.zeros((1, cfg.E)), W, W, logits_in=logits)
    st = fw["stats"]
    assert st[oracle.ST_DROPPED] == ex["dropped"]
    np.testing.assert_allclose(st[oracle.ST_PBAR:], [_frac(v) for v in ex["pbar"]], rtol=1e-14)
    assert st[oracle.ST_AUX_LOSS] == pytest.approx(_frac(ex["aux_loss"]), rel=1e-12)
    assert st[oracle.ST_AUX_SWITCH] == pytest.approx(_frac(ex["aux_switch"]), rel=1e-12)
    assert st[oracle.ST_MAX_OVER_MEAN_KEPT] == pytest.approx(_frac(ex["max_over_mean_kept"]))
    assert st[oracle.ST_COUNT_CV] == pytest.approx(_frac(ex["count_cv"]))
    assert st[oracle.ST_MAX_OVER_MEAN_COUNT] == pytest.approx(_frac(ex["max_over_mean_count"]))


def test_capacity_values_of_the_workloads(oracle_lib):
    # C = ceil(cf * T * k / E) with the fp32 factor 1.2f:
    # 1.2*2048*2/4 = 1228.8 -> 1229; 1.2*16384*2/8 = 4915.2 -> 4916; 1.2*65536*2/16 = 9830.4 -> 9831
    cf = float(np.float32(1.2))
    for (T, E, want) in ((2048, 4, 1229), (16384, 8, 4916), (65536, 16, 9831)):
        assert oracle.capacity(oracle.OracleConfig(T=T, d=1, f=1, E=E, k=2, capacity_factor=cf)) == want
    # no factor -> each expert may see every token once
    assert oracle.capacity(oracle.OracleConfig(T=77, d=1, f=1, E=4, k=2)) == 77
    # clamped to T
    assert oracle.capacity(oracle.OracleConfig(T=10, d=1, f=1, E=2, k=2, capacity_factor=50.0)) == 10


# --------------------------------------------------------------------------- brute force
@pytest.mark.parametrize("swiglu", [False, True])
@pytest.mark.parametrize("cf", [0.0, 1.0, 0.5])
@pytest.mark.parametrize("norm", [True, False])
def test_matches_bruteforce_mask_loop(oracle_lib, swiglu, cf, norm):
    rng = np.random.default_rng(1234 + int(swiglu) + int(cf * 10) + int(norm))
    T, d, f, E, k = 37, 12, 20, 5, 2
    x, Wr, Wup, Wg, Wd, b, nz = _rand_case(rng, T, d, f, E, k, swiglu, bias=True, noise=True)
    cfg = oracle.OracleConfig(T=T, d=d, f=f, E=E, k=k, capacity_factor=cf, swiglu=swiglu,
                              normalize_gates=norm, pad_m=4)
    r = oracle.forward(cfg, x, Wr, Wup, Wd, Wgate=Wg, bias=b, noise=nz)
    out, topk, gate, kept = bruteforce.forward(x, Wr, Wup, Wd, k, cf, Wgate=Wg, bias=b, noise=nz,
                                               normalize_gates=norm)
    assert (r["topk_idx"] == topk).all()
    np.testing.assert_allclose(r["gate"], gate, rtol=1e-13, atol=0)
    assert ((r["slot_of"] >= 0) == kept).all()
    np.testing.assert_allclose(r["out"], out, rtol=1e-12, atol=1e-13)


def test_topk_against_full_sort_with_ties_and_nan(oracle_lib):
    rng = np.random.default_rng(7)
    T, E = 300, 8
    logits = rng.integers(-3, 4, size=(T, E)).astype(np.float64)  # many exact ties
    logits[::17, 3] = np.nan
    logits[::23, :] = 1.0                                          # all tied
    for k in (1, 2, 3, 8):
        cfg = oracle.OracleConfig(T=T, d=1, f=1, E=E, k=k)
        r = oracle.route(cfg, logits)
        assert (r["topk_idx"] == bruteforce.topk_by_sort(logits, k)).all()
        assert r["nonfinite"] == int(np.isnan(logits).any(axis=1).sum())


# --------------------------------------------------------------------------- closed forms
def test_single_expert_is_a_plain_ffn(oracle_lib):
    rng = np.random.default_rng(3)
    T, d, f = 9, 7, 11
    x = rng.standard_normal((T, d))
    Wup = rng.standard_normal((1, d, f))
    Wd = rng.standard_normal((1, f, d))
    cfg = oracle.OracleConfig(T=T, d=d, f=f, E=1, k=1)
    r = oracle.forward(cfg, x, rng.standard_normal((d, 1)), Wup, Wd)
    h = x @ Wup[0]
    want = (h / (1 + np.exp(-h))) @ Wd[0]
    np.testing.assert_allclose(r["out"], want, rtol=1e-12, atol=1e-12)
    assert (r["gate"] == 1.0).all()


def test_k_equals_E_is_a_dense_softmax_mixture(oracle_lib):
    rng = np.random.default_rng(4)
    T, d, f, E = 6, 5, 8, 3
    x, Wr, Wup, Wg, Wd, _, _ = _rand_case(rng, T, d, f, E, E, swiglu=True)
    cfg = oracle.OracleConfig(T=T, d=d, f=f, E=E, k=E, swiglu=True)
    r = oracle.forward(cfg, x, Wr, Wup, Wd, Wgate=Wg)
    z = x @ Wr
    p = np.exp(z - z.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    want = np.zeros((T, d))
    for e in range(E):
        g = x @ Wg[e]
        want += p[:, e:e + 1] * (((g / (1 + np.exp(-g))) * (x @ Wup[e])) @ Wd[e])
    np.testing.assert_allclose(r["out"], want, rtol=1e-12, atol=1e-12)


def test_uniform_router_aux_statistics(oracle_lib):
    T, d, E, k = 64, 4, 8, 2
    cfg = oracle.OracleConfig(T=T, d=d, f=2, E=E, k=k, aux_coef=0.01)
    x = np.random.default_rng(5).standard_normal((T, d))
    r = oracle.forward(cfg, x, np.zeros((d, E)), np.zeros((E, d, 2)), np.zeros((E, 2, d)))
    st = r["stats"]
    np.testing.assert_allclose(st[oracle.ST_PBAR:], 1.0 / E, rtol=1e-15)
    assert st[oracle.ST_AUX_LOSS] == pytest.approx(0.0, abs=1e-18)
    assert st[oracle.ST_AUX_SWITCH] == pytest.approx(1.0, rel=1e-14)
    assert st[oracle.ST_ENTROPY] == pytest.approx(math.log(E), rel=1e-14)
    # all logits tie -> every token picks experts 0 and 1
    assert (r["topk_idx"] == [0, 1]).all()


# --------------------------------------------------------------------------- invariants
@pytest.mark.parametrize("cf", [0.0, 1.2, 0.7])
def test_routing_invariants(oracle_lib, cf):
    rng = np.random.default_rng(11)
    T, E, k, pad = 500, 6, 2, 8
    logits = rng.standard_normal((T, E)) + np.array([1.5, 0.8, 0, 0, -0.5, -1.0])
    cfg = oracle.OracleConfig(T=T, d=1, f=1, E=E, k=k, capacity_factor=cf, pad_m=pad)
    r = oracle.route(cfg, logits)
    p = oracle.permute(cfg, r["topk_idx"])
    topk, slot = r["topk_idx"], p["slot_of"]
    C = oracle.capacity(cfg)
    # k distinct experts per token; gates sum to one before drops
    assert all(len(set(row)) == k for row in topk.tolist())
    np.testing.assert_allclose(r["gate"].sum(1), 1.0, rtol=1e-14)
    assert r["counts"].sum() == T * k
    assert (p["kept"] == np.minimum(r["counts"], C)).all()
    dropped = int((slot < 0).sum())
    assert p["kept"].sum() == T * k - dropped
    off = p["offsets"]
    assert off[0] == 0 and ((np.diff(off) % pad) == 0).all()
    assert (np.diff(off) - p["kept"] < pad).all() and (np.diff(off) >= p["kept"]).all()
    perm = p["perm_token"]
    for e in range(E):
        seg = perm[off[e]:off[e + 1]]
        real = seg[: p["kept"][e]]
        assert (np.diff(real) > 0).all()                       # ascending token order
        assert (seg[p["kept"][e]:] == -1).all()                # padding rows
        want = [t for t in range(T) if e in topk[t]][:C]       # first C in token order
        assert real.tolist() == want
    for t in range(T):
        for j in range(k):
            if slot[t, j] >= 0:
                assert perm[slot[t, j]] == t
                assert off[topk[t, j]] <= slot[t, j] < off[topk[t, j] + 1]


# --------------------------------------------------------------------------- gradients
def _loss(cfg, x, Wr, Wup, Wd, Wg, b, nz, dout):
    r = oracle.forward(cfg, x, Wr, Wup, Wd, Wgate=Wg, bias=b, noise=nz)
    return float((dout * r["out"]).sum() + r["stats"][oracle.ST_AUX_LOSS]), r


@pytest.mark.parametrize("swiglu,cf,norm", [(False, 0.0, True), (False, 0.75, True),
                                            (True, 0.0, True), (True, 0.75, False),
                                            (False, 0.0, False)])
def test_backward_matches_finite_differences(oracle_lib, swiglu, cf, norm):
    rng = np.random.default_rng(100 + int(swiglu) * 10 + int(cf * 4) + int(norm))
    T, d, f, E, k = 8, 8, 16, 4, 2
    x, Wr, Wup, Wg, Wd, b, nz = _rand_case(rng, T, d, f, E, k, swiglu, bias=True, noise=True)
    dout = rng.standard_normal((T, d))
    cfg = oracle.OracleConfig(T=T, d=d, f=f, E=E, k=k, capacity_factor=cf, swiglu=swiglu,
                              normalize_gates=norm, aux_coef=0.3)
    L0, r0 = _loss(cfg, x, Wr, Wup, Wd, Wg, b, nz, dout)
    g = oracle.backward(cfg, x, Wr, Wup, Wd, r0["logits"], r0["topk_idx"], r0["gate"],
                        r0["slot_of"], dout, Wgate=Wg, with_bias=True)
    h = 1e-6
    params = {"x": (x, g["dx"]), "Wr": (Wr, g["dWr"]), "b": (b, g["db"]),
              "Wup": (Wup, g["dWup"]), "Wd": (Wd, g["dWdown"])}
    if swiglu:
        params["Wg"] = (Wg, g["dWgate"])
    checked = 0
    for name, (arr, grad) in params.items():
        idxs = [np.unravel_index(i, arr.shape) for i in
                rng.choice(arr.size, size=min(arr.size, 40), replace=False)]
        for ix in idxs:
            vals = []
            for s in (+h, -h):
                a2 = arr.copy()
                a2[ix] += s
                kw = dict(x=x, Wr=Wr, Wup=Wup, Wd=Wd, Wg=Wg, b=b, nz=nz)
                kw[name] = a2
                L, r = _loss(cfg, kw["x"], kw["Wr"], kw["Wup"], kw["Wd"], kw["Wg"], kw["b"],
                             kw["nz"], dout)
                assert (r["topk_idx"] == r0["topk_idx"]).all(), "routing moved under +-h"
                assert (r["slot_of"] == r0["slot_of"]).all()
                vals.append(L)
            fd = (vals[0] - vals[1]) / (2 * h)
            assert grad[ix] == pytest.approx(fd, rel=2e-5, abs=2e-7), (name, ix)
            checked += 1
    assert checked > 150


def test_backward_gate_gradient_is_dot_with_expert_output(oracle_lib):
    """dL/dgate[t,j] = <dout_t, FFN_{e_j}(x_t)> for kept slots, 0 for dropped ones."""
    rng = np.random.default_rng(9)
    T, d, f, E, k = 10, 6, 9, 3, 2
    x, Wr, Wup, Wg, Wd, _, _ = _rand_case(rng, T, d, f, E, k)
    cfg = oracle.OracleConfig(T=T, d=d, f=f, E=E, k=k, capacity_factor=0.5)
    r = oracle.forward(cfg, x, Wr, Wup, Wd)
    dout = rng.standard_normal((T, d))
    g = oracle.backward(cfg, x, Wr, Wup, Wd, r["logits"], r["topk_idx"], r["gate"],
                        r["slot_of"], dout)
    for t in range(T):
        for j in range(k):
            if r["slot_of"][t, j] < 0:
                assert g["dgate"][t, j] == 0.0
            else:
                y = oracle.expert_apply(cfg, r["topk_idx"][t, j], x[t], Wup, None, Wd)
                assert g["dgate"][t, j] == pytest.approx(float(dout[t] @ y), rel=1e-12)


def test_backward_on_a_token_sample_matches_the_full_batch_rows(oracle_lib):
    """Per-token gradients of a sampled sub-batch, with the full batch's pbar and T
    for the aux term, equal those rows of the full-batch backward."""
    rng = np.random.default_rng(21)
    T, d, f, E, k = 40, 6, 10, 4, 2
    x, Wr, Wup, Wg, Wd, b, nz = _rand_case(rng, T, d, f, E, k, swiglu=True, bias=True, noise=True)
    cfg = oracle.OracleConfig(T=T, d=d, f=f, E=E, k=k, capacity_factor=0.8, swiglu=True,
                              aux_coef=0.2)
    r = oracle.forward(cfg, x, Wr, Wup, Wd, Wgate=Wg, bias=b, noise=nz)
    dout = rng.standard_normal((T, d))
    full = oracle.backward(cfg, x, Wr, Wup, Wd, r["logits"], r["topk_idx"], r["gate"],
                           r["slot_of"], dout, Wgate=Wg)
    idx = np.array([0, 3, 17, 39])
    sub = oracle.OracleConfig(T=len(idx), d=d, f=f, E=E, k=k, capacity_factor=0.8, swiglu=True,
                              aux_coef=0.2)
    part = oracle.backward(sub, x[idx], Wr, Wup, Wd, r["logits"][idx], r["topk_idx"][idx],
                           r["gate"][idx], r["slot_of"][idx], dout[idx], Wgate=Wg,
                           pbar=r["stats"][oracle.ST_PBAR:], T_aux=T)
    for key in ("dx", "dlogits", "dgate"):
        np.testing.assert_allclose(part[key], full[key][idx], rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------- router variants
@pytest.mark.parametrize("tau,st,masked,norm", [(0.6, False, False, True), (1.7, False, True, False),
                                                (0.7, True, False, True), (0.7, True, True, True)])
def test_router_variants_match_bruteforce(oracle_lib, tau, st, masked, norm):
    """Temperature, straight-through (Gumbel) top-k and padding masks agree with
    the brute-force restatement ([Twinkle] §3.1; [LLaMA4-MoE] §4.1)."""
    rng = np.random.default_rng(int(tau * 10) + 2 * st + 4 * masked)
    T, d, f, E, k = 41, 10, 14, 6, 2
    x, Wr, Wup, Wg, Wd, b, nz = _rand_case(rng, T, d, f, E, k, bias=True, noise=True)
    nz = -np.log(-np.log(rng.uniform(1e-9, 1.0, (T, E)))) if st else nz   # Gumbel draws
    mask = (rng.uniform(size=T) > 0.3).astype(np.uint8) if masked else None
    cfg = oracle.OracleConfig(T=T, d=d, f=f, E=E, k=k, capacity_factor=0.8, normalize_gates=norm,
                              temperature=tau, straight_through=st, aux_coef=0.1, pad_m=4)
    r = oracle.forward(cfg, x, Wr, Wup, Wd, bias=b, noise=nz, mask=mask)
    out, topk, gate, kept = bruteforce.forward(x, Wr, Wup, Wd, k, 0.8, bias=b, noise=nz,
                                               normalize_gates=norm, temperature=tau,
                                               straight_through=st, mask=mask)
    assert (r["topk_idx"] == topk).all()
    np.testing.assert_allclose(r["gate"], gate, rtol=1e-13, atol=0)
    assert ((r["slot_of"] >= 0) == kept).all()
    np.testing.assert_allclose(r["out"], out, rtol=1e-12, atol=1e-13)
    if masked:
        assert r["stats"][oracle.ST_TOKENS] == mask.sum()
        assert (r["topk_idx"][mask == 0] == -1).all() and (r["out"][mask == 0] == 0).all()
    if st:
        assert (r["gate"][r["topk_idx"] >= 0] == 1.0).all()


def test_temperature_backward_matches_finite_differences(oracle_lib):
    rng = np.random.default_rng(77)
    T, d, f, E, k = 8, 6, 12, 4, 2
    x, Wr, Wup, Wg, Wd, b, nz = _rand_case(rng, T, d, f, E, k, bias=True, noise=True)
    dout = rng.standard_normal((T, d))
    for norm in (True, False):
        cfg = oracle.OracleConfig(T=T, d=d, f=f, E=E, k=k, normalize_gates=norm, aux_coef=0.3,
                                  temperature=0.7)
        L0, r0 = _loss(cfg, x, Wr, Wup, Wd, None, b, nz, dout)
        g = oracle.backward(cfg, x, Wr, Wup, Wd, r0["logits"], r0["topk_idx"], r0["gate"],
                            r0["slot_of"], dout, with_bias=True)
        h = 1e-6
        for name, arr, grad in (("Wr", Wr, g["dWr"]), ("b", b, g["db"]), ("x", x, g["dx"])):
            for ix in [np.unravel_index(i, arr.shape) for i in range(0, arr.size, max(1, arr.size // 12))]:
                vals = []
                for s in (+h, -h):
                    a2 = arr.copy()
                    a2[ix] += s
                    kw = dict(x=x, Wr=Wr, b=b)
                    kw[name] = a2
                    L, r = _loss(cfg, kw["x"], kw["Wr"], Wup, Wd, None, kw["b"], nz, dout)
                    assert (r["topk_idx"] == r0["topk_idx"]).all()
                    vals.append(L)
                assert grad[ix] == pytest.approx((vals[0] - vals[1]) / (2 * h), rel=2e-5, abs=2e-7)


def test_straight_through_gradient_is_the_surrogate_derivative(oracle_lib):
    """Straight-through Gumbel top-k ([Twinkle] §3.1): forward gates are 1; the
    router gradient is that of the surrogate sum_j dgate_j p_{e_j}(logits/tau)
    plus the aux loss, at fixed selection.  The expert-weight gradients are exact."""
    rng = np.random.default_rng(88)
    T, d, f, E, k, tau = 9, 6, 10, 5, 2, 0.7
    x, Wr, Wup, Wg, Wd, b, _ = _rand_case(rng, T, d, f, E, k, bias=True)
    gum = -np.log(-np.log(rng.uniform(1e-9, 1.0, (T, E))))
    dout = rng.standard_normal((T, d))
    cfg = oracle.OracleConfig(T=T, d=d, f=f, E=E, k=k, aux_coef=0.2, temperature=tau,
                              straight_through=True)
    r = oracle.forward(cfg, x, Wr, Wup, Wd, bias=b, noise=gum)
    g = oracle.backward(cfg, x, Wr, Wup, Wd, r["logits"], r["topk_idx"], r["gate"], r["slot_of"],
                        dout, with_bias=True)
    topk, dg = r["topk_idx"], g["dgate"]

    def surrogate(logits):
        z = logits / tau
        p = np.exp(z - z.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        pbar = p.mean(0)
        return float((dg * np.take_along_axis(p, topk, 1)).sum() + 0.2 * ((pbar - 1 / E) ** 2).sum())

    h = 1e-6
    for t in range(T):
        for e in range(E):
            lp, lm = r["logits"].copy(), r["logits"].copy()
            lp[t, e] += h
            lm[t, e] -= h
            fd = (surrogate(lp) - surrogate(lm)) / (2 * h)
            assert g["dlogits"][t, e] == pytest.approx(fd, rel=1e-6, abs=1e-9)
    # expert weights: exact derivative of <dout, out> (gates are constants 1)
    L0, _ = _loss(cfg, x, Wr, Wup, Wd, None, b, gum, dout)
    for ix in [(0, 1, 2), (1, 0, 3), (3, 5, 1)]:
        for arr_name in ("Wup", "Wd"):
            arr = Wup if arr_name == "Wup" else Wd
            grad = g["dWup"] if arr_name == "Wup" else g["dWdown"]
            vals = []
            for s in (+h, -h):
                a2 = arr.copy()
                a2[ix] += s
                L, _ = _loss(cfg, x, Wr, a2 if arr_name == "Wup" else Wup,
                             a2 if arr_name == "Wd" else Wd, None, b, gum, dout)
                vals.append(L)
            assert grad[ix] == pytest.approx((vals[0] - vals[1]) / (2 * h), rel=2e-5, abs=2e-7)


def test_masked_batch_equals_the_batch_without_padding(oracle_lib):
    """Padding tokens take no part in routing ([LLaMA4-MoE] §4.1): outputs,
    statistics and gradients equal those of the real tokens alone."""
    rng = np.random.default_rng(99)
    T, d, f, E, k = 30, 8, 12, 4, 2
    x, Wr, Wup, Wg, Wd, b, _ = _rand_case(rng, T, d, f, E, k, swiglu=True, bias=True)
    mask = (rng.uniform(size=T) > 0.35).astype(np.uint8)
    real = np.nonzero(mask)[0]
    dout = rng.standard_normal((T, d))
    full = oracle.OracleConfig(T=T, d=d, f=f, E=E, k=k, swiglu=True, aux_coef=0.3, temperature=0.9)
    sub = oracle.OracleConfig(T=len(real), d=d, f=f, E=E, k=k, swiglu=True, aux_coef=0.3,
                              temperature=0.9)
    rf = oracle.forward(full, x, Wr, Wup, Wd, Wgate=Wg, bias=b, mask=mask)
    rs = oracle.forward(sub, x[real], Wr, Wup, Wd, Wgate=Wg, bias=b)
    np.testing.assert_allclose(rf["out"][real], rs["out"], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(rf["stats"][oracle.ST_PBAR:], rs["stats"][oracle.ST_PBAR:], rtol=1e-13)
    for i in (oracle.ST_AUX_LOSS, oracle.ST_AUX_SWITCH, oracle.ST_ENTROPY, oracle.ST_TOKENS):
        assert rf["stats"][i] == pytest.approx(rs["stats"][i], rel=1e-13)
    gf = oracle.backward(full, x, Wr, Wup, Wd, rf["logits"], rf["topk_idx"], rf["gate"],
                         rf["slot_of"], dout, Wgate=Wg, with_bias=True)
    gs = oracle.backward(sub, x[real], Wr, Wup, Wd, rs["logits"], rs["topk_idx"], rs["gate"],
                         rs["slot_of"], dout[real], Wgate=Wg, with_bias=True)
    np.testing.assert_allclose(gf["dx"][real], gs["dx"], rtol=1e-12, atol=1e-14)
    assert (gf["dx"][mask == 0] == 0).all()
    for key in ("dWr", "db", "dWup", "dWgate", "dWdown"):
        np.testing.assert_allclose(gf[key], gs[key], rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------- shared experts
def _shared_case(rng, d, fs, swiglu):
    return (rng.standard_normal((d, fs)) * 0.3, rng.standard_normal((fs, d)) * 0.3,
            rng.standard_normal((d, fs)) * 0.3 if swiglu else None)


@pytest.mark.parametrize("swiglu,cf,masked", [(False, 0.0, False), (True, 0.75, False),
                                              (False, 0.6, True)])
def test_shared_experts_match_bruteforce(oracle_lib, swiglu, cf, masked):
    rng = np.random.default_rng(500 + int(swiglu) + 2 * int(masked))
    T, d, f, E, k, fs = 40, 12, 10, 5, 2, 24
    x, Wr, Wup, Wg, Wd, b, _ = _rand_case(rng, T, d, f, E, k, swiglu, bias=True)
    Wus, Wds, Wgs = _shared_case(rng, d, fs, swiglu)
    mask = (rng.random(T) > 0.3).astype(np.uint8) if masked else None
    cfg = oracle.OracleConfig(T=T, d=d, f=f, E=E, k=k, capacity_factor=cf, swiglu=swiglu,
                              f_shared=fs)
    r = oracle.forward(cfg, x, Wr, Wup, Wd, Wgate=Wg, bias=b, mask=mask, Wup_s=Wus, Wdown_s=Wds,
                       Wgate_s=Wgs)
    out, topk, _, _ = bruteforce.forward(x, Wr, Wup, Wd, k, cf, Wgate=Wg, bias=b, mask=mask,
                                         shared=(Wus, Wds, Wgs))
    assert (r["topk_idx"] == topk).all()
    np.testing.assert_allclose(r["out"], out, rtol=1e-11, atol=1e-11)
    if masked:   # padding tokens skip the routed experts, not the shared ones
        pad = mask == 0
        sh = bruteforce.forward(x, Wr, Wup, Wd, k, cf, Wgate=Wg, bias=b,
                                mask=np.zeros(T, np.uint8), shared=(Wus, Wds, Wgs))[0]
        np.testing.assert_allclose(r["out"][pad], sh[pad], rtol=1e-11, atol=1e-11)


def test_shared_expert_equal_to_the_routed_one_doubles_a_plain_ffn(oracle_lib):
    """E = k = 1 routes every token to expert 0 with gate 1; a shared FFN with
    the same weights adds the same FFN once more: out = 2 W_d^T silu(W_u^T x)."""
    rng = np.random.default_rng(7)
    T, d, f = 9, 7, 11
    x = rng.standard_normal((T, d))
    Wup = rng.standard_normal((1, d, f))
    Wd = rng.standard_normal((1, f, d))
    cfg = oracle.OracleConfig(T=T, d=d, f=f, E=1, k=1, f_shared=f)
    r = oracle.forward(cfg, x, rng.standard_normal((d, 1)), Wup, Wd, Wup_s=Wup[0], Wdown_s=Wd[0])
    h = x @ Wup[0]
    np.testing.assert_allclose(r["out"], 2 * (h / (1 + np.exp(-h))) @ Wd[0], rtol=1e-12,
                               atol=1e-12)


def test_shared_experts_side_by_side_are_one_wide_ffn(oracle_lib):
    """Two shared experts of width f, run as straight-through experts that every
    token selects (E = k = 2, gates 1), equal one shared FFN of width 2f whose
    weight blocks are the two experts' side by side."""
    rng = np.random.default_rng(8)
    T, d, f = 10, 6, 9
    x = rng.standard_normal((T, d))
    Wup = rng.standard_normal((2, d, f)) * 0.5
    Wg = rng.standard_normal((2, d, f)) * 0.5
    Wd = rng.standard_normal((2, f, d)) * 0.5
    Wr = rng.standard_normal((d, 2))
    two = oracle.forward(oracle.OracleConfig(T=T, d=d, f=f, E=2, k=2, swiglu=True,
                                             straight_through=True), x, Wr, Wup, Wd, Wgate=Wg)
    assert (two["gate"] == 1.0).all()
    # a layer whose routed experts are all zero, plus the wide shared FFN
    cfg = oracle.OracleConfig(T=T, d=d, f=f, E=2, k=1, swiglu=True, f_shared=2 * f)
    z = np.zeros_like(Wup)
    wide = oracle.forward(cfg, x, Wr, z, z, Wgate=z, Wup_s=np.concatenate([Wup[0], Wup[1]], 1),
                          Wgate_s=np.concatenate([Wg[0], Wg[1]], 1),
                          Wdown_s=np.concatenate([Wd[0], Wd[1]], 0))
    np.testing.assert_allclose(wide["out"], two["out"], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("swiglu,cf", [(False, 0.75), (True, 0.0)])
def test_shared_expert_backward_matches_finite_differences(oracle_lib, swiglu, cf):
    rng = np.random.default_rng(600 + int(swiglu))
    T, d, f, E, k, fs = 8, 8, 16, 4, 2, 12
    x, Wr, Wup, Wg, Wd, b, nz = _rand_case(rng, T, d, f, E, k, swiglu, bias=True, noise=True)
    Wus, Wds, Wgs = _shared_case(rng, d, fs, swiglu)
    dout = rng.standard_normal((T, d))
    cfg = oracle.OracleConfig(T=T, d=d, f=f, E=E, k=k, capacity_factor=cf, swiglu=swiglu,
                              aux_coef=0.3, f_shared=fs)

    def loss(kw):
        r = oracle.forward(cfg, kw["x"], Wr, Wup, Wd, Wgate=Wg, bias=b, noise=nz,
                           Wup_s=kw["Wus"], Wdown_s=kw["Wds"], Wgate_s=kw["Wgs"])
        return float((dout * r["out"]).sum() + r["stats"][oracle.ST_AUX_LOSS]), r

    base = dict(x=x, Wus=Wus, Wds=Wds, Wgs=Wgs)
    L0, r0 = loss(base)
    g = oracle.backward(cfg, x, Wr, Wup, Wd, r0["logits"], r0["topk_idx"], r0["gate"],
                        r0["slot_of"], dout, Wgate=Wg, Wup_s=Wus, Wdown_s=Wds, Wgate_s=Wgs)
    params = {"x": g["dx"], "Wus": g["dWup_s"], "Wds": g["dWdown_s"]}
    if swiglu:
        params["Wgs"] = g["dWgate_s"]
    h, checked = 1e-6, 0
    for name, grad in params.items():
        arr = base[name]
        for i in rng.choice(arr.size, size=min(arr.size, 40), replace=False):
            ix = np.unravel_index(i, arr.shape)
            vals = []
            for s in (+h, -h):
                kw = dict(base)
                kw[name] = arr.copy()
                kw[name][ix] += s
                L, r = loss(kw)
                assert (r["slot_of"] == r0["slot_of"]).all(), "routing moved under +-h"
                vals.append(L)
            assert grad[ix] == pytest.approx((vals[0] - vals[1]) / (2 * h), rel=2e-5, abs=2e-7)
            checked += 1
    assert checked >= 120


# --------------------------------------------------------------------------- single dW entries
def _kept_tokens(cfg, r, e):
    """Expert e's kept (token, gate) pairs in ascending token order."""
    tt, jj = np.nonzero((r["topk_idx"] == e) & (r["slot_of"] >= 0))
    order = np.argsort(tt, kind="stable")
    return tt[order], r["gate"][tt[order], jj[order]]


@pytest.mark.parametrize("swiglu,cf,norm,st", [(False, 0.75, False, False), (True, 0.0, True, False),
                                               (True, 0.8, True, False), (False, 0.0, True, True)])
def test_wgrad_entries_equal_the_full_backward(oracle_lib, swiglu, cf, norm, st):
    """Every entry of dW_up / dW_gate / dW_down from the per-entry definition
    equals the full-matrix backward (capacity drops, raw gates, straight-through
    gates of 1 included)."""
    rng = np.random.default_rng(300 + 10 * int(swiglu) + int(cf * 4) + 2 * int(norm) + int(st))
    T, d, f, E, k = 24, 8, 12, 4, 2
    x, Wr, Wup, Wg, Wd, b, nz = _rand_case(rng, T, d, f, E, k, swiglu, bias=True, noise=True)
    dout = rng.standard_normal((T, d))
    cfg = oracle.OracleConfig(T=T, d=d, f=f, E=E, k=k, capacity_factor=cf, swiglu=swiglu,
                              normalize_gates=norm, aux_coef=0.3, straight_through=st)
    r = oracle.forward(cfg, x, Wr, Wup, Wd, Wgate=Wg, bias=b, noise=nz)
    if cf > 0:
        assert (r["slot_of"] < 0).any(), "the case should drop assignments"
    g = oracle.backward(cfg, x, Wr, Wup, Wd, r["logits"], r["topk_idx"], r["gate"], r["slot_of"],
                        dout, Wgate=Wg, with_bias=True)
    jj, ii = np.meshgrid(np.arange(f), np.arange(d), indexing="ij")   # [f, d] grids
    for e in range(E):
        toks, gates = _kept_tokens(cfg, r, e)
        kinds = [(oracle.WGRAD_DOWN, jj.ravel(), ii.ravel(), g["dWdown"][e]),
                 (oracle.WGRAD_UP, ii.T.ravel(), jj.T.ravel(), g["dWup"][e])]
        if swiglu:
            kinds.append((oracle.WGRAD_GATE, ii.T.ravel(), jj.T.ravel(), g["dWgate"][e]))
        for kind, rows, cols, full in kinds:
            got = oracle.expert_wgrad_entries(cfg, x[toks], gates, dout[toks], Wup[e], Wd[e],
                                              np.full(len(rows), kind), rows, cols,
                                              Wg_e=Wg[e] if swiglu else None)
            want = full[rows, cols]
            np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def test_wgrad_entries_match_finite_differences(oracle_lib):
    """Single entries against central differences of <dout, out> + aux loss in
    the expert weights (SwiGLU, capacity drops): pinned to the loss itself."""
    rng = np.random.default_rng(401)
    T, d, f, E, k = 10, 6, 8, 3, 2
    x, Wr, Wup, Wg, Wd, b, nz = _rand_case(rng, T, d, f, E, k, swiglu=True, bias=True)
    dout = rng.standard_normal((T, d))
    cfg = oracle.OracleConfig(T=T, d=d, f=f, E=E, k=k, capacity_factor=0.8, swiglu=True,
                              aux_coef=0.3)
    L0, r0 = _loss(cfg, x, Wr, Wup, Wd, Wg, b, nz, dout)
    h = 1e-6
    checked = 0
    for name, kind in (("Wd", oracle.WGRAD_DOWN), ("Wup", oracle.WGRAD_UP),
                       ("Wg", oracle.WGRAD_GATE)):
        for _ in range(12):
            e = int(rng.integers(E))
            if name == "Wd":
                rr, cc = int(rng.integers(f)), int(rng.integers(d))
            else:
                rr, cc = int(rng.integers(d)), int(rng.integers(f))
            vals = []
            for s in (+h, -h):
                kw = dict(x=x, Wr=Wr, Wup=Wup, Wd=Wd, Wg=Wg, b=b, nz=nz)
                a2 = kw[name].copy()
                a2[e, rr, cc] += s
                kw[name] = a2
                L, r = _loss(cfg, kw["x"], kw["Wr"], kw["Wup"], kw["Wd"], kw["Wg"], kw["b"],
                             kw["nz"], dout)
                assert (r["slot_of"] == r0["slot_of"]).all()
                vals.append(L)
            fd = (vals[0] - vals[1]) / (2 * h)
            toks, gates = _kept_tokens(cfg, r0, e)
            got = oracle.expert_wgrad_entries(cfg, x[toks], gates, dout[toks], Wup[e], Wd[e],
                                              [kind], [rr], [cc], Wg_e=Wg[e])[0]
            assert got == pytest.approx(fd, rel=2e-5, abs=2e-7), (name, e, rr, cc)
            checked += 1
    assert checked == 36
