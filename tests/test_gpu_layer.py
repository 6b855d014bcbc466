"""GPU parity of the whole layer through the C ABI against the fp64 oracle."""
import json

import numpy as np
import pytest
import torch

import moe_inputs
import top_routing_expert_moe_gb300 as moe
from tests import parity

pytestmark = pytest.mark.gpu


def _w(name, **kw):
    from dataclasses import replace
    w = moe_inputs.get(name)
    return replace(w, **kw) if kw else w


def _report(name, rep):
    print(f"\n[{name}] " + json.dumps({k: (round(v, 8) if isinstance(v, float) else v)
                                       for k, v in rep.items()}))


@pytest.mark.parametrize("pad_m", [1, 8, 128])
def test_tiny_fp32_full(pad_m):
    w = _w("tiny_fp32")
    inp = moe_inputs.make_inputs(w, 0)
    rep, _ = parity.full_check(w, inp, pad_m=pad_m, backward=True)
    _report(f"tiny_fp32 pad{pad_m}", rep)


def test_small_bf16_full():
    w = _w("small_bf16")
    inp = moe_inputs.make_inputs(w, 0)
    rep, _ = parity.full_check(w, inp, sample_rows=512)
    _report("small_bf16", rep)


def test_llama4_shape_reduced_tokens():
    w = _w("llama4_bf16").with_tokens(1024)
    inp = moe_inputs.make_inputs(w, 0)
    rep, _ = parity.full_check(w, inp, sample_rows=256)
    _report(w.name, rep)


def test_skewed16_shape_reduced_tokens():
    w = _w("skewed16_bf16").with_tokens(1024)
    inp = moe_inputs.make_inputs(w, 0)
    rep, r = parity.full_check(w, inp, sample_rows=256)
    assert rep and r["layer"].stats[4].item() > 0, "the skewed workload should drop tokens"
    _report(w.name, rep)


def test_mixtral_shape_reduced_tokens():
    w = _w("mixtral_bf16").with_tokens(128)
    inp = moe_inputs.make_inputs(w, 0)
    rep, _ = parity.full_check(w, inp, sample_rows=64)
    _report(w.name, rep)


# ------------------------------------------------------------------ edge cases
def _edge_inputs(w, seed=3):
    return moe_inputs.make_inputs(w, seed)


def test_ragged_tokens_and_raw_gates_fp32():
    w = _w("tiny_fp32", T=301, capacity_factor=0.9)
    rep, _ = parity.full_check(w, _edge_inputs(w), pad_m=4, normalize=False)
    _report("ragged_raw_fp32", rep)


def test_ragged_tokens_bf16_top1():
    w = _w("small_bf16", T=333, k=1, d=256, f=384)
    rep, _ = parity.full_check(w, _edge_inputs(w))
    _report("ragged_top1_bf16", rep)


def test_odd_dwr_unit_count_bf16():
    """d = 384 and 200 tokens: 3 column chunks x 13 token chunks of dW_r, an odd
    number of 128-thread units, so the last CTA of the router-backward launch runs
    one unit and its other half returns at once; d also gives three 128-row blocks
    in dW_up."""
    w = _w("small_bf16", T=200, d=384, f=256)
    rep, _ = parity.full_check(w, _edge_inputs(w, seed=61))
    _report("odd_dwr_units_bf16", rep)


def test_k_equals_E_bf16():
    w = _w("small_bf16", T=200, E=4, k=4, d=256, f=256, capacity_factor=0.0)
    rep, _ = parity.full_check(w, _edge_inputs(w))
    _report("k_eq_E_bf16", rep)


def test_empty_expert_and_exact_capacity_bf16():
    """Expert 3 never selected (bias -1e4); expert 0 over capacity (bias +1e4)."""
    w = _w("small_bf16", T=256, d=256, f=256, capacity_factor=1.0)
    inp = _edge_inputs(w)
    inp["bias"] = np.array([1e4, 0.0, 0.0, -1e4], np.float32)
    rep, r = parity.full_check(w, inp)
    kept = r["layer"].kept.cpu().numpy()
    assert kept[3] == 0 and kept[0] == 128      # C = ceil(1.0*256*2/4) = 128
    _report("empty_and_capped_bf16", rep)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_exact_ties_lowest_id_wins(dtype):
    """Router columns 4 and 5 duplicate columns 1 and 2.  The GPU's own logits
    of each pair must be bit-identical (so the tie really reaches the top-k),
    and the lower expert id must win it: 4 / 5 are never a token's first pick,
    and a token whose first pick is 1 (2) takes 4 (5) second, the tied pair in
    id order.  Everything else is checked bit-exact against the oracle."""
    if dtype == "fp32":
        w = _w("tiny_fp32", T=130, E=6, k=2)
        pad_m = 2
    else:
        w = _w("small_bf16", T=384, d=256, f=256, E=6, k=2, capacity_factor=0.0)
        pad_m = 128
    inp = _edge_inputs(w)
    Wr = inp["W_r"].copy()
    Wr[:, 4] = Wr[:, 1]
    Wr[:, 5] = Wr[:, 2]
    inp["W_r"] = Wr
    rep, r = parity.full_check(w, inp, pad_m=pad_m)
    lg = r["layer"].logits
    assert torch.equal(lg[:, 4], lg[:, 1]) and torch.equal(lg[:, 5], lg[:, 2]), \
        "duplicated router columns did not give bit-identical logits"
    topk = r["layer"].topk_idx.cpu().numpy()
    assert not np.isin(topk[:, 0], [4, 5]).any()
    first1, first2 = topk[:, 0] == 1, topk[:, 0] == 2
    assert first1.sum() + first2.sum() >= w.T // 8, "too few tokens meet an exact tie"
    assert (topk[first1, 1] == 4).all() and (topk[first2, 1] == 5).all()
    rep["tied_first_picks"] = int(first1.sum() + first2.sum())
    _report(f"exact_ties_{dtype}", rep)


def _guarded(shape, dtype, guard=4096, fill=0xA5):
    """A tensor of `shape` placed inside a larger byte buffer whose `guard`
    bytes before and after it (and the tensor itself) hold the byte `fill`."""
    n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
    buf = torch.full((n + 2 * guard,), fill, dtype=torch.uint8, device="cuda")
    return buf, buf[guard:guard + n].view(dtype).view(*shape)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_outputs_stay_inside_their_buffers(dtype):
    """Canary guards around every output of the forward and backward entry
    points (a stand-in for an out-of-bounds checker): after the layer ran, the
    guard bytes before and after each output still hold the sentinel, the rows
    the layout leaves unused (at and past offsets[E] in the permuted buffers)
    are untouched too, and the results equal an unguarded run byte for byte."""
    if dtype == "bf16":
        w = _w("small_bf16", T=333, d=256, f=384, E=4, k=2, capacity_factor=1.0)
        pad_m = 128
    else:
        w = _w("tiny_fp32", T=301, d=64, f=96, E=5, k=2, capacity_factor=0.9)
        pad_m = 8
    inp = _edge_inputs(w, seed=71)
    ref = parity.run_gpu(w, inp, pad_m=pad_m)
    assert ref["status"] == 0
    cfg = parity.gpu_cfg(w, pad_m)
    dt, tdt = w.dtype, cfg.torch_dtype
    T, d, f, E, k, R, nh = w.T, w.d, w.f, w.E, w.k, ref["layer"].rows_cap, cfg.nh
    x, Wr = parity.to_torch(inp["x"], dt), parity.to_torch(inp["W_r"], dt)
    Wu, Wd = parity.to_torch(inp["W_up"], dt), parity.to_torch(inp["W_down"], dt)
    Wg = parity.to_torch(inp.get("W_gate"), dt)
    dout = parity.to_torch(inp["dout"], dt)
    i32, f32 = torch.int32, torch.float32
    shapes = dict(logits=((T, E), f32), topk=((T, k), i32), gate=((T, k), f32),
                  counts=((E,), i32), stats=((9 + E,), f32), x_perm=((R, d), tdt),
                  perm_token=((R,), i32), slot_of=((T, k), i32), kept=((E,), i32),
                  offsets=((E + 1,), i32), h=((nh, R, f), tdt), act=((R, f), tdt),
                  y=((R, d), tdt), out=((T, d), tdt), dy=((R, d), tdt), dgate=((T, k), f32),
                  dh=((nh, R, f), tdt), dxp=((R, d), tdt), dlogits=((T, E), f32),
                  dx=((T, d), tdt), dWr=((d, E), tdt), dWu=((E, d, f), tdt),
                  dWd=((E, f, d), tdt), ws=((moe.workspace_size(cfg),), torch.uint8))
    bufs, t = {}, {}
    for name, (shape, tt) in shapes.items():
        bufs[name], t[name] = _guarded(shape, tt)
    moe.moe_route(cfg, x, Wr, None, None, None, t["logits"], t["topk"], t["gate"], t["counts"],
                  t["stats"], t["ws"])
    moe.moe_permute(cfg, x, t["topk"], t["x_perm"], t["perm_token"], t["slot_of"], t["kept"],
                    t["offsets"], t["stats"], t["ws"])
    moe.moe_grouped_ffn(cfg, t["x_perm"], t["offsets"], Wu, Wg, Wd, t["h"], t["act"], t["y"],
                        t["ws"])
    moe.moe_combine(cfg, t["y"], t["slot_of"], t["gate"], t["out"])
    moe.moe_combine_backward(cfg, dout, t["y"], t["gate"], t["slot_of"], t["perm_token"],
                             t["offsets"], t["dy"], t["dgate"])
    moe.moe_grouped_ffn_backward(cfg, t["x_perm"], t["offsets"], Wu, Wg, Wd, t["h"], t["act"],
                                 t["dy"], t["dh"], t["dxp"], t["dWu"], None, t["dWd"], t["ws"])
    moe.moe_router_backward(cfg, x, Wr, t["logits"], t["topk"], t["gate"], t["slot_of"],
                            t["dgate"], t["dxp"], t["stats"], t["dx"], t["dWr"], None,
                            t["dlogits"], t["ws"])
    torch.cuda.synchronize()
    assert moe.last_device_status() == 0
    for name, b in bufs.items():
        g = 4096
        assert (b[:g] == 0xA5).all() and (b[-g:] == 0xA5).all(), f"write outside {name}"
    rows = int(t["offsets"][-1].item())
    assert 0 < rows < R
    for name in ("x_perm", "act", "y", "dy", "dxp"):
        assert (t[name][rows:].view(torch.uint8) == 0xA5).all(), f"{name}: rows past offsets[E]"
    for name in ("h", "dh"):
        assert (t[name][:, rows:].contiguous().view(torch.uint8) == 0xA5).all(), name
    assert (t["perm_token"][rows:].view(torch.uint8) == 0xA5).all()
    L, g = ref["layer"], ref["grads"]
    same = dict(logits=L.logits, topk=L.topk_idx, gate=L.gate, counts=L.counts,
                offsets=L.offsets, slot_of=L.slot_of, kept=L.kept, out=L.out, dx=g["dx"],
                dWr=g["dW_r"], dWu=g["dW_up"], dWd=g["dW_down"], dgate=ref["dgate"],
                dlogits=ref["dlogits"])
    for name, want in same.items():
        assert torch.equal(t[name], want), name
    for name, want in (("x_perm", L.x_perm), ("act", L.act), ("y", L.y_perm),
                       ("dy", ref["dy"]), ("dxp", ref["dxp"])):
        assert torch.equal(t[name][:rows], want[:rows]), name


def test_reruns_are_bit_identical():
    w = _w("small_bf16", T=512)
    inp = moe_inputs.make_inputs(w, 1)
    a = parity.run_gpu(w, inp)
    outs_a = [t.clone() for t in (a["layer"].out, a["grads"]["dx"], a["grads"]["dW_up"],
                                  a["grads"]["dW_down"], a["grads"]["dW_r"])]
    b = parity.run_gpu(w, inp)
    outs_b = [b["layer"].out, b["grads"]["dx"], b["grads"]["dW_up"], b["grads"]["dW_down"],
              b["grads"]["dW_r"]]
    for x, y in zip(outs_a, outs_b):
        assert torch.equal(x, y)


def test_composite_backward_matches_substeps():
    w = _w("small_bf16", T=512)
    inp = moe_inputs.make_inputs(w, 2)
    r = parity.run_gpu(w, inp)
    L = r["layer"]
    sub = {k: v.clone() for k, v in r["grads"].items() if v is not None}
    g = L.backward(r["dout"])
    torch.cuda.synchronize()
    for k, v in sub.items():
        if k == "dbias":
            continue
        assert torch.equal(v, g[k]), k


def test_nonfinite_logits_are_flagged():
    import top_routing_expert_moe_gb300 as moe
    w = _w("tiny_fp32", T=64)
    inp = moe_inputs.make_inputs(w, 0)
    inp["x"][5, 0] = np.nan
    r = parity.run_gpu(w, inp, backward=False)
    assert r["status"] == moe.ERR_NONFINITE
    assert r["layer"].stats[moe.STAT_NONFINITE].item() == 1.0
    assert moe.last_device_status() == 0   # reading clears it


@pytest.mark.parametrize("E,k,dtype", [(1, 1, "bf16"), (1, 1, "fp32"), (2, 1, "bf16"),
                                       (8, 1, "bf16"), (12, 3, "bf16"),
                                       (16, 4, "bf16"), (32, 2, "bf16"), (48, 4, "bf16"),
                                       (64, 2, "bf16"), (64, 8, "bf16"),
                                       (12, 3, "fp32"), (64, 5, "fp32")])
def test_expert_count_and_top_k_sweep(E, k, dtype):
    """Top-k / expert-count sweep (top-1 routing, wide k, up to 64 experts, expert counts
    that are not powers of two: padded expert slots in the router and its backward)."""
    base = "small_bf16" if dtype == "bf16" else "tiny_fp32"
    w = _w(base, T=640, E=E, k=k, d=256 if dtype == "bf16" else 64,
           f=256 if dtype == "bf16" else 96, capacity_factor=1.1)
    rep, _ = parity.full_check(w, _edge_inputs(w, seed=E * 10 + k),
                               pad_m=128 if dtype == "bf16" else 8)
    _report(f"sweep E{E} k{k} {dtype}", rep)


@pytest.mark.parametrize("T,dtype", [(1, "bf16"), (3, "bf16"), (17, "bf16"), (1, "fp32"),
                                     (5, "fp32")])
def test_decode_sized_batches(T, dtype):
    """A handful of tokens (decode-sized batches): one partly filled router tile, most
    experts empty, weight gradients reduced over one or two rows."""
    base = "small_bf16" if dtype == "bf16" else "tiny_fp32"
    w = _w(base, T=T, d=256 if dtype == "bf16" else 64, f=256 if dtype == "bf16" else 96,
           E=8, k=2, capacity_factor=0.0)
    rep, r = parity.full_check(w, _edge_inputs(w, seed=40 + T), pad_m=128 if dtype == "bf16" else 8)
    assert int(r["layer"].kept.sum().item()) == 2 * T
    _report(f"decode batch T{T} {dtype}", rep)


@pytest.mark.parametrize("cf,dtype", [(0.001, "bf16"), (0.0625, "bf16"), (0.001, "fp32")])
def test_extreme_capacity(cf, dtype):
    """Capacity 1 (cf = 0.001) and 10 (cf = 0.0625) per expert at 640 tokens, 8 experts, top-2:
    nearly every assignment dropped, most tokens lose both slots (zero output rows), and the
    backward reduces over a handful of kept rows."""
    base = "small_bf16" if dtype == "bf16" else "tiny_fp32"
    w = _w(base, T=640, d=256 if dtype == "bf16" else 64, f=256 if dtype == "bf16" else 96,
           E=8, k=2, capacity_factor=cf)
    rep, r = parity.full_check(w, _edge_inputs(w, seed=77), pad_m=128 if dtype == "bf16" else 8)
    C = moe.capacity(parity.gpu_cfg(w))
    assert C == (1 if cf < 0.01 else 10)
    kept = r["layer"].kept.cpu().numpy()
    assert (kept <= C).all() and kept.sum() <= 8 * C
    assert (r["layer"].slot_of.cpu().numpy() < 0).all(1).sum() > 0   # fully dropped tokens exist
    _report(f"extreme capacity cf{cf} {dtype}", rep)


# ------------------------------------------------------------------ router variants
@pytest.mark.parametrize("tau,normalize,dtype", [(0.5, True, "bf16"), (2.0, False, "bf16"),
                                                 (0.7, True, "fp32"), (3.0, False, "fp32")])
def test_softmax_temperature(tau, normalize, dtype):
    base = "small_bf16" if dtype == "bf16" else "tiny_fp32"
    w = _w(base, T=777, d=256 if dtype == "bf16" else 64, f=256 if dtype == "bf16" else 96,
           E=8, k=2, capacity_factor=1.25)
    rep, _ = parity.full_check(w, _edge_inputs(w, seed=11), pad_m=128 if dtype == "bf16" else 4,
                               normalize=normalize, temperature=tau)
    _report(f"temperature {tau} norm{int(normalize)} {dtype}", rep)


@pytest.mark.parametrize("dtype,E,k,tau", [("bf16", 8, 2, 1.0), ("bf16", 16, 4, 0.5),
                                           ("fp32", 6, 1, 2.0)])
def test_straight_through_gumbel_topk(dtype, E, k, tau):
    """Selection on logits + Gumbel draws, gates 1, gradient through softmax(l / tau)."""
    base = "small_bf16" if dtype == "bf16" else "tiny_fp32"
    w = _w(base, T=640, d=256 if dtype == "bf16" else 64, f=256 if dtype == "bf16" else 96,
           E=E, k=k, capacity_factor=1.3)
    inp = _edge_inputs(w, seed=21)
    inp["noise"] = moe_inputs.gumbel(21, w.T, w.E)
    rep, r = parity.full_check(w, inp, pad_m=128 if dtype == "bf16" else 8,
                               temperature=tau, straight_through=True)
    assert (r["layer"].gate == 1).all()
    # the draws change the selection relative to the noise-free logits
    plain = np.argsort(-parity.np64(r["layer"].logits), axis=1, kind="stable")[:, :k]
    assert (np.sort(plain, 1) != np.sort(r["layer"].topk_idx.cpu().numpy(), 1)).any(1).mean() > 0.2
    _report(f"straight-through E{E} k{k} tau{tau} {dtype}", rep)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_padding_tokens_take_no_part(dtype):
    base = "small_bf16" if dtype == "bf16" else "tiny_fp32"
    w = _w(base, T=1100, d=256 if dtype == "bf16" else 64, f=256 if dtype == "bf16" else 96,
           E=8, k=2, capacity_factor=1.1)
    inp = _edge_inputs(w, seed=31)
    inp["mask"] = moe_inputs.padding_mask(31, w.T)
    rep, r = parity.full_check(w, inp, pad_m=128 if dtype == "bf16" else 4)
    L = r["layer"]
    pad = inp["mask"] == 0
    assert pad.sum() > 128
    assert (L.topk_idx.cpu().numpy()[pad] == -1).all()
    assert (L.out.float().cpu().numpy()[pad] == 0).all()
    assert (r["grads"]["dx"].float().cpu().numpy()[pad] == 0).all()
    assert L.stats[moe.STAT_TOKENS].item() == int((~pad).sum())
    _report(f"padding mask {dtype}", rep)


def test_padding_mask_with_noise_temperature_and_raw_gates():
    w = _w("llama4_bf16").with_tokens(1024)
    inp = moe_inputs.make_inputs(w, 4)
    inp["mask"] = moe_inputs.padding_mask(4, w.T, seq_len=256)
    rep, _ = parity.full_check(w, inp, sample_rows=256, normalize=False, temperature=1.5)
    _report("llama4 mask+noise+tau", rep)


def test_every_token_padding():
    w = _w("small_bf16", T=300, d=256, f=256)
    inp = _edge_inputs(w, seed=41)
    inp["mask"] = np.zeros(w.T, np.uint8)
    rep, r = parity.full_check(w, inp)
    L = r["layer"]
    assert int(L.offsets[-1].item()) == 0 and int(L.counts.sum().item()) == 0
    for name in ("dx", "dW_up", "dW_down", "dW_r"):
        assert (r["grads"][name].float() == 0).all(), name
    _report("all padding", rep)


# ------------------------------------------------------------------ shared experts
@pytest.mark.parametrize("dtype,swiglu,T,fs", [("bf16", False, 333, 384), ("bf16", True, 256, 256),
                                               ("fp32", False, 150, 96), ("fp32", True, 97, 40)])
def test_shared_experts(dtype, swiglu, T, fs):
    """Routed experts plus a shared FFN on every token (weight 1), in the same
    GEMM launches; ragged T leaves zero rows past T in the shared buffers."""
    base = "small_bf16" if dtype == "bf16" else "tiny_fp32"
    w = _w(base, T=T, d=256 if dtype == "bf16" else 64, f=256 if dtype == "bf16" else 96,
           E=6, k=2, capacity_factor=1.0, swiglu=swiglu, f_shared=fs)
    rep, _ = parity.full_check(w, _edge_inputs(w, seed=51), pad_m=128 if dtype == "bf16" else 4)
    assert "y_shared_rel" in rep and "dWup_s_rel" in rep
    _report(f"shared {dtype} swiglu{int(swiglu)} T{T} fs{fs}", rep)


def test_shared_experts_with_padding_and_llama4_shape():
    w = _w("llama4_bf16", f_shared=1024).with_tokens(512)
    inp = moe_inputs.make_inputs(w, 6)
    inp["mask"] = moe_inputs.padding_mask(6, w.T)
    rep, _ = parity.full_check(w, inp, sample_rows=128)
    _report("llama4 + shared + mask", rep)


def test_shared_experts_composite_backward_matches_substeps():
    w = _w("small_bf16", T=384, d=256, f=256, f_shared=512)
    inp = moe_inputs.make_inputs(w, 7)
    r = parity.run_gpu(w, inp)
    L = r["layer"]
    sub = {k: v.clone() for k, v in r["grads"].items() if v is not None}
    g = L.backward(r["dout"])
    torch.cuda.synchronize()
    for k, v in sub.items():
        if k == "dbias":
            continue
        assert torch.equal(v, g[k]), k


@pytest.mark.parametrize("T", [384, 8192])   # one tile and many
def test_out_of_range_expert_index_is_reported(T):
    """An expert index outside [0, E) in a caller's top-k (a bad input to moe_permute) is
    caught by the permutation kernels' own bounds checks: the device status reads
    MOE_ERR_DEVICE_BOUNDS and the entry is dropped exactly as a -1 (no selection) there
    would be — the permutation is byte-identical to that run, which reports nothing."""
    E, k, d = 8, 2, 256
    cfg = moe.MoEConfig(T=T, d=d, f=256, E=E, k=k, capacity_factor=1.25, dtype=moe.BF16,
                        pad_m=128)
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(T)
    topk = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    bad_t, bad_j = T // 3, 1
    x = torch.randn(T, d, generator=g).to(torch.bfloat16).to(dev)
    rows = moe.rows_capacity(cfg)
    ws = torch.empty(moe.workspace_size(cfg), dtype=torch.uint8, device=dev)

    def run(fill):
        tk = topk.clone()
        tk[bad_t, bad_j] = fill
        tk = tk.to(dev)
        out = dict(x_perm=torch.empty(rows, d, dtype=torch.bfloat16, device=dev),
                   perm_token=torch.empty(rows, dtype=torch.int32, device=dev),
                   slot_of=torch.empty(T, k, dtype=torch.int32, device=dev),
                   kept=torch.empty(E, dtype=torch.int32, device=dev),
                   offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   stats=torch.zeros(9 + E, dtype=torch.float32, device=dev))
        moe.last_device_status()              # start from a clear status word
        moe.moe_permute(cfg, x, tk, out["x_perm"], out["perm_token"], out["slot_of"], out["kept"],
                        out["offsets"], out["stats"], ws)
        status = moe.last_device_status()     # reading clears it
        n = int(out["offsets"][E].item())
        out["x_perm"] = out["x_perm"][:n]
        out["perm_token"] = out["perm_token"][:n]
        return status, out

    st_bad, bad = run(E + 5)
    st_none, none = run(-1)
    assert st_bad == moe.ERR_DEVICE_BOUNDS and st_none == 0
    assert int(bad["slot_of"][bad_t, bad_j].item()) == -1
    for key in ("slot_of", "kept", "offsets", "perm_token", "x_perm"):
        assert torch.equal(bad[key], none[key]), key
    assert torch.equal(bad["stats"][moe.STAT_DROPPED], none["stats"][moe.STAT_DROPPED])
