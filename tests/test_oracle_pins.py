"""Pins of the CPU oracle to things other than itself (CPU only).

Each ``check_*`` takes the oracle module, so the same checks can be re-run on the oracle with
one planted mistake: ``test_planted_mistakes_are_caught`` shows that a dropped term, a wrong
index, a transposed operand or a wrong rounding rule fails a pin.
"""
import json
from fractions import Fraction
import math
import os

import numpy as np
import pytest
import scipy.special as sps
import torch
import torch.nn.functional as F

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


# ----------------------------------------------------------------------------- checks
def check_router(o):
    # library routine: torch's Linear without bias, on a non-square shape
    x = RNG.standard_normal((5, 7))
    w = RNG.standard_normal((3, 7))
    ref = F.linear(torch.from_numpy(x), torch.from_numpy(w)).numpy()
    np.testing.assert_allclose(o.router_logits(x, w), ref, rtol=1e-13, atol=1e-13)
    # hand case: x = (1, 2, 3), rows of W_r pick x1 and x2 + x3
    z = o.router_logits(np.array([[1.0, 2.0, 3.0]]), np.array([[1.0, 0, 0], [0, 1.0, 1.0]]))
    assert z.tolist() == [[1.0, 5.0]]
    # the fixed logit bias shifts only its own column
    zb = o.router_logits(x, w, np.array([2.0, 0.0, 0.0]))
    np.testing.assert_allclose(zb - ref, np.tile([2.0, 0.0, 0.0], (5, 1)), atol=1e-13)


def check_softmax(o):
    z = RNG.standard_normal((9, 6)) * 3
    P, lse = o.softmax_lse(z)
    assert np.all(np.abs(P.sum(1) - 1) <= 1e-12)
    np.testing.assert_allclose(P, sps.softmax(z, axis=1), rtol=1e-13)
    np.testing.assert_allclose(lse, sps.logsumexp(z, axis=1), rtol=1e-13)
    P2, lse2 = o.softmax_lse(np.array([[0.0, math.log(3.0)]]))
    np.testing.assert_allclose(P2, [[0.25, 0.75]], rtol=1e-14)
    np.testing.assert_allclose(lse2, [math.log(4.0)], rtol=1e-14)
    P0, lse0 = o.softmax_lse(np.zeros((2, 8)))
    assert np.all(P0 == 1.0 / 8) and np.allclose(lse0, math.log(8.0), rtol=1e-15)


def check_topk(o):
    # explicit tie cases
    assert o.topk_select(np.array([[1.0, 3.0, 3.0, 0.0]]), 2).tolist() == [[1, 2]]
    assert o.topk_select(np.array([[2.0, 2.0]]), 1).tolist() == [[0]]
    assert o.topk_select(np.array([[0.0, 5.0, 1.0, 5.0]]), 3).tolist() == [[1, 3, 2]]
    # brute force: full Python sort by (-z, e) on tiny integer logits (many exact ties)
    for T, E, k in [(64, 8, 2), (40, 5, 5), (30, 4, 1), (25, 8, 6)]:
        z = RNG.integers(-2, 3, size=(T, E)).astype(np.float64)
        got = o.topk_select(z, k)
        for t in range(T):
            ref = sorted(range(E), key=lambda e: (-z[t, e], e))[:k]
            assert got[t].tolist() == ref, (t, z[t])
        gap = o.topk_gap(z, k)
        for t in range(T):
            zs = sorted(z[t], reverse=True)
            assert gap[t] == (math.inf if k == E else zs[k - 1] - zs[k])


def check_renormalise(o):
    z = RNG.standard_normal((20, 8))
    P, _ = o.softmax_lse(z)
    idx = o.topk_select(z, 3)
    w = o.renormalise(P, idx)
    assert np.all(np.abs(w.sum(1) - 1) <= 1e-12)
    # equals the softmax over the selected logits (the GPT-4 article's form)
    np.testing.assert_allclose(w, sps.softmax(np.take_along_axis(z, idx, 1), axis=1), rtol=1e-12)


def check_capacity(o):
    assert o.capacity(1.25, 8192, 2, 16) == 1280
    assert o.capacity(1.0, 16384, 2, 128) == 256
    assert o.capacity(1.0, 10, 1, 3) == 4          # ceil(10/3)
    assert o.capacity(0.5, 3, 1, 1) == 2           # ceil(1.5)
    assert o.capacity(0.1, 10, 1, 1) == 2          # float32(0.1) > 0.1, so 10 cf > 1
    assert o.capacity(0.0, 10, 2, 4) is None and o.capacity(-1.0, 10, 2, 4) is None


def _brute_dispatch(idx, E, cap):
    T, k = idx.shape
    per = [[(t, j) for t in range(T) for j in range(k) if idx[t, j] == e] for e in range(E)]
    kept = [p if cap is None else p[:cap] for p in per]
    rows = [a for e in range(E) for a in kept[e]]
    return per, kept, rows


def check_dispatch(o):
    for T, E, k, cap in [(50, 6, 2, None), (50, 6, 2, 7), (33, 4, 3, 1), (16, 8, 8, 2), (1, 3, 1, 1)]:
        z = RNG.standard_normal((T, E))
        z[:, 0] += 1.5   # skew so that capacity bites
        idx = o.topk_select(z, k)
        lay = o.dispatch(idx, E, cap)
        per, kept, rows = _brute_dispatch(idx, E, cap)
        assert lay["counts"].tolist() == [len(p) for p in per]
        assert int(lay["counts"].sum()) == T * k
        assert lay["kept_counts"].tolist() == [len(p) for p in kept]
        assert int(lay["kept_counts"].sum()) == T * k - lay["drops"]
        if cap is not None:
            assert lay["kept_counts"].tolist() == [min(len(p), cap) for p in per]
        assert lay["offsets"].tolist() == [0] + list(np.cumsum([len(p) for p in kept]))
        assert lay["tok_of"].tolist() == [t for (t, _) in rows]
        for r, (t, j) in enumerate(rows):
            assert lay["row_of"][t, j] == r
        n_kept = int((lay["row_of"] >= 0).sum())
        assert n_kept == len(rows)
        for e in range(E):
            toks = lay["tok_of"][lay["offsets"][e]:lay["offsets"][e + 1]]
            assert np.all(np.diff(toks) > 0)


def check_activations(o):
    u = np.linspace(-9, 9, 1001)
    np.testing.assert_allclose(o.gelu_erf(u), F.gelu(torch.from_numpy(u)).numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(o.silu(u), F.silu(torch.from_numpy(u)).numpy(), rtol=1e-12, atol=1e-15)
    assert o.gelu_erf(np.array([0.0]))[0] == 0.0 and o.silu(np.array([0.0]))[0] == 0.0
    assert abs(o.gelu_erf(np.array([1.0]))[0] - 0.5 * (1 + math.erf(1 / math.sqrt(2)))) < 1e-15


def _torch_ffn(xr, act, w_up, w_down, w_gate=None, b_up=None, b_down=None):
    t = lambda a: None if a is None else torch.as_tensor(np.asarray(a, np.float64))
    x = t(xr)
    if act == "gelu":
        h = F.gelu(F.linear(x, t(w_up), t(b_up)))
    else:
        h = F.silu(F.linear(x, t(w_gate))) * F.linear(x, t(w_up))
    return F.linear(h, t(w_down), t(b_down)).numpy()


def check_expert_ffn(o):
    d, f = 12, 20
    xr = RNG.standard_normal((7, d))
    wu, wd, wg = RNG.standard_normal((f, d)), RNG.standard_normal((d, f)), RNG.standard_normal((f, d))
    bu, bd = RNG.standard_normal(f), RNG.standard_normal(d)
    np.testing.assert_allclose(o.expert_ffn(xr, "gelu", wu, wd, None, bu, bd),
                               _torch_ffn(xr, "gelu", wu, wd, None, bu, bd), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(o.expert_ffn(xr, "swiglu", wu, wd, wg),
                               _torch_ffn(xr, "swiglu", wu, wd, wg), rtol=1e-11, atol=1e-11)


def _identical_expert_inputs(T, d, E, f, act, S=0, bias=True):
    x = RNG.standard_normal((T, d))
    wr = RNG.standard_normal((E, d))
    wu, wd, wg = RNG.standard_normal((f, d)), RNG.standard_normal((d, f)), RNG.standard_normal((f, d))
    bu, bd = RNG.standard_normal(f), RNG.standard_normal(d)
    rep = lambda a: np.repeat(a[None], E, 0)
    inp = dict(x=x, w_router=wr, logit_bias=None, w_up=rep(wu), w_down=rep(wd),
               w_gate=rep(wg) if act == "swiglu" else None,
               b_up=rep(bu) if (bias and act == "gelu") else None,
               b_down=rep(bd) if (bias and act == "gelu") else None)
    if S:
        inp.update(ws_up=np.repeat(wu[None], S, 0), ws_down=np.repeat(wd[None], S, 0),
                   ws_gate=np.repeat(wg[None], S, 0) if act == "swiglu" else None)
    dense = _torch_ffn(x, act, wu, wd, wg if act == "swiglu" else None,
                       inp["b_up"][0] if inp["b_up"] is not None else None,
                       inp["b_down"][0] if inp["b_down"] is not None else None)
    return inp, dense


def check_layer_reductions(o):
    # k = E with identical experts: the renormalised weights sum to 1, so y is one dense FFN
    for act in ("gelu", "swiglu"):
        inp, dense = _identical_expert_inputs(T=24, d=10, E=4, f=16, act=act)
        out = o.moe_layer(inp, E=4, k=4, act=act)
        np.testing.assert_allclose(out["y"], dense, rtol=1e-10, atol=1e-10)
    # E = 1, k = 1: a dense FFN
    inp, dense = _identical_expert_inputs(T=9, d=8, E=1, f=8, act="gelu")
    np.testing.assert_allclose(o.moe_layer(inp, E=1, k=1, act="gelu")["y"], dense, rtol=1e-10, atol=1e-10)
    # shared experts identical to the routed ones, no biases: y = (1 + S) dense FFN
    inp, dense = _identical_expert_inputs(T=11, d=8, E=3, f=16, act="swiglu", S=2, bias=False)
    np.testing.assert_allclose(o.moe_layer(inp, E=3, k=2, act="swiglu", n_shared=2)["y"], 3 * dense,
                               rtol=1e-10, atol=1e-10)
    # capacity: all tokens forced onto expert 0 with k = 1 and cap = 3; later tokens get nothing
    inp, dense = _identical_expert_inputs(T=10, d=6, E=3, f=8, act="gelu")
    inp["logit_bias"] = np.array([1e3, 0.0, 0.0])
    out = o.moe_layer(inp, E=3, k=1, act="gelu", cf=0.9)  # cap = ceil(0.9 * 10 / 3) = 3
    assert out["cap"] == 3 and out["drops"] == 7
    np.testing.assert_allclose(out["y"][:3], dense[:3], rtol=1e-10, atol=1e-10)
    assert np.all(out["y"][3:] == 0)
    # subset evaluation equals the rows of the full evaluation
    inp, _ = _identical_expert_inputs(T=15, d=6, E=5, f=8, act="gelu")
    inp["w_up"] = RNG.standard_normal(inp["w_up"].shape)
    full = o.moe_layer(inp, E=5, k=2, act="gelu")
    sub = o.moe_layer(inp, E=5, k=2, act="gelu", tokens=[3, 0, 14])
    np.testing.assert_allclose(sub["y"], full["y"][[3, 0, 14]], rtol=1e-13, atol=1e-13)


def _frac(a):
    a = np.asarray(a, dtype=np.float64)
    return a[..., 0] / a[..., 1]


def check_combine_fixture(o):
    # hand-worked fixture (tests/golden/combine_distinct_experts.json): three experts with distinct
    # constant outputs, k = 2, so the pairing of each slot's weight with its expert's row shows
    g = json.load(open(os.path.join(GOLDEN, "combine_distinct_experts.json")))
    E, k = g["E"], g["k"]
    x = np.log(np.asarray(g["x_as_log"], np.float64))
    c = np.asarray(g["c"], np.float64)
    T, d = x.shape
    inp = dict(x=x, w_router=np.eye(E, d), logit_bias=None,
               w_up=np.zeros((E, 1, d)), b_up=np.zeros((E, 1)), w_down=np.zeros((E, d, 1)), b_down=c.copy())
    out = o.moe_layer(inp, E=E, k=k, act="gelu", lb_coef=0.01)
    assert out["idx"].tolist() == g["topk_idx"]
    np.testing.assert_allclose(out["w"], _frac(g["topk_w"]), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(out["y"], _frac(g["y_dropless"]), rtol=1e-13, atol=1e-13)
    assert abs(out["lb"] - 0.01 * g["lb_over_alpha"]) < 1e-15
    cap = o.moe_layer(inp, E=E, k=k, act="gelu", cf=g["capacity_factor"])
    assert cap["cap"] == g["capacity"]
    assert cap["row_of"].tolist() == g["row_of_capped"]
    assert cap["kept_counts"].tolist() == g["kept_capped"]
    np.testing.assert_allclose(cap["y"], _frac(g["y_capped"]), rtol=1e-13, atol=1e-13)
    # per-token brute force on random distinct experts (k = 3 of E = 5, SwiGLU, shared expert,
    # capacity drops): y_t = sum over kept slots of w_tj FFN_{e_tj}(x_t) + FFN_shared(x_t),
    # evaluated token by token without the expert-sorted layout
    T, d, E, k, f = 23, 6, 5, 3, 8
    inp = dict(x=RNG.standard_normal((T, d)), w_router=RNG.standard_normal((E, d)), logit_bias=None,
               w_gate=RNG.standard_normal((E, f, d)), w_up=RNG.standard_normal((E, f, d)),
               w_down=RNG.standard_normal((E, d, f)), ws_gate=RNG.standard_normal((1, f, d)),
               ws_up=RNG.standard_normal((1, f, d)), ws_down=RNG.standard_normal((1, d, f)))
    out = o.moe_layer(inp, E=E, k=k, act="swiglu", n_shared=1, cf=0.8)
    assert out["drops"] > 0
    z = inp["x"] @ inp["w_router"].T
    for t in range(T):
        sel = sorted(range(E), key=lambda e: (-z[t, e], e))[:k]
        p = np.exp(z[t] - z[t].max())
        p = p / p.sum()
        yt = _torch_ffn(inp["x"][t:t + 1], "swiglu", inp["ws_up"][0], inp["ws_down"][0], inp["ws_gate"][0])[0]
        for j, e in enumerate(sel):
            if out["row_of"][t, j] >= 0:
                yt = yt + p[e] / p[sel].sum() * _torch_ffn(inp["x"][t:t + 1], "swiglu", inp["w_up"][e],
                                                            inp["w_down"][e], inp["w_gate"][e])[0]
        np.testing.assert_allclose(out["y"][t], yt, rtol=1e-10, atol=1e-10)


def check_losses(o):
    E, T, k = 8, 32, 2
    # zero router weights: every Pbar_e = 1/E exactly, so lb = alpha for any counts; zl = beta (ln E)^2
    P, lse = o.softmax_lse(np.zeros((T, E)))
    for counts in (np.full(E, T * k // E), np.array([T * k] + [0] * (E - 1))):
        lb, zl = o.aux_losses(P, lse, counts, k, 0.01, 0.001)
        assert abs(lb - 0.01) < 1e-15
        assert abs(zl - 0.001 * math.log(E) ** 2) < 1e-15
    assert abs(o.lb_loss_squared_mean_form(P, 0.01) - 0.01) < 1e-15
    # two experts, every assignment on expert 0, Pbar = (p, 1-p): lb = alpha * 2 * p
    z = np.array([[math.log(3.0), 0.0]] * 4)     # P = (3/4, 1/4)
    P, lse = o.softmax_lse(z)
    lb, zl = o.aux_losses(P, lse, np.array([4, 0]), 1, 0.5, 1.0)
    assert abs(lb - 0.5 * 2 * 0.75) < 1e-14
    assert abs(zl - math.log(4.0) ** 2) < 1e-14
    assert o.aux_losses(np.zeros((0, 4)), np.zeros(0), np.zeros(4), 2, 0.01, 0.001) == (0.0, 0.0)


def check_coactivation(o):
    # hand-worked fixture (tests/golden/coactivation_small.json)
    g = json.load(open(os.path.join(GOLDEN, "coactivation_small.json")))
    idx = np.array(g["topk_idx"])
    C = o.coactivation(idx, g["E"])
    assert C.tolist() == g["coact"]
    S = o.coactivation_score(C)
    assert abs(S[0, 1] - g["score_0_to_1"]) < 1e-15 and abs(S[2, 1] - g["score_2_to_1"]) < 1e-15
    offsets = np.array([0, 0, 0, 0, g["kept"]])
    imb, drop = o.routing_stats(idx, g["E"], g["k"], offsets)
    assert abs(imb - g["imbalance"]) < 1e-15 and abs(drop - g["dropped_fraction"]) < 1e-15
    # invariants on random top-k selections: symmetric, diagonal = counts, each token choosing i
    # has k - 1 other (distinct) experts, all pairs add up to T k (k - 1)
    for T, E, k in [(50, 8, 2), (37, 6, 3), (20, 5, 5), (30, 4, 1)]:
        idx = o.topk_select(RNG.standard_normal((T, E)), k)
        C = o.coactivation(idx, E)
        assert (C == C.T).all()
        assert (np.diag(C) == np.bincount(idx.ravel(), minlength=E)).all()
        off = C.sum(1) - np.diag(C)
        assert (off == (k - 1) * np.diag(C)).all()
        assert C.sum() - np.trace(C) == T * k * (k - 1)
        if k == E:
            assert (C == T).all()
        if k == 1:
            assert (C - np.diag(np.diag(C)) == 0).all()
        imb, drop = o.routing_stats(idx, E, k)
        assert imb >= 1.0 - 1e-12 and drop == 0.0
    assert o.routing_stats(np.zeros((0, 2), dtype=int), 4, 2) == (0.0, 0.0)
    # router entropy: the definition -sum P ln P directly (scipy's entropy), uniform logits give
    # ln E, a near one-hot router ~0, two experts the binary entropy of sigmoid(z_0 - z_1)
    z = RNG.standard_normal((40, 7)) * 2
    P, _ = o.softmax_lse(z)
    assert abs(o.router_entropy(z) - float(np.mean(sps.entr(P).sum(axis=1)))) < 1e-12
    assert abs(o.router_entropy(np.zeros((5, 6))) - math.log(6)) < 1e-14
    hot = np.zeros((3, 4))
    hot[:, 2] = 60.0
    assert o.router_entropy(hot) < 1e-20
    z2 = RNG.standard_normal((25, 2))
    p = sps.expit(z2[:, 0] - z2[:, 1])
    assert abs(o.router_entropy(z2) - float(np.mean(-p * np.log(p) - (1 - p) * np.log(1 - p)))) < 1e-12
    assert o.router_entropy(np.zeros((0, 3))) == 0.0
    # the GPT-4 2% article's balance form: torch's kl_div (target uniform, log of the smoothed mean
    # probabilities, summed) plus the squared frequency gap; zero at exactly uniform routing
    z = RNG.standard_normal((30, 5))
    P, _ = o.softmax_lse(z)
    counts = np.array([20, 15, 10, 10, 5])
    ref_kl = torch.nn.functional.kl_div(torch.log(torch.tensor(P.mean(axis=0)) + 1e-8),
                                        torch.full((5,), 0.2, dtype=torch.float64), reduction="sum").item()
    ref = 0.01 * (ref_kl + float(np.sum((counts / counts.sum() - 0.2) ** 2)))
    assert abs(o.lb_loss_kl_frequency_form(P, counts, 0.01) - ref) < 1e-15
    assert abs(o.lb_loss_kl_frequency_form(np.full((4, 5), 0.2), np.full(5, 3), 0.5, eps=0.0)) < 1e-15
    # all tokens to one expert (k = 1): frequency term (E - 1) / E
    assert abs(o.lb_loss_kl_frequency_form(np.full((4, 5), 0.2), np.array([4, 0, 0, 0, 0]), 1.0, eps=0.0)
               - 0.8) < 1e-15


def _bwd_case(rng, T, d, E, k, dff, act, bias, n_shared, wscale=0.7):
    """Small layer whose top-k margins are far above a finite-difference step."""
    while True:
        inp = dict(x=rng.standard_normal((T, d)), w_router=rng.standard_normal((E, d)) * wscale,
                   w_up=rng.standard_normal((E, dff, d)) * 0.5, w_down=rng.standard_normal((E, d, dff)) * 0.5)
        if act == "swiglu":
            inp["w_gate"] = rng.standard_normal((E, dff, d)) * 0.5
        if bias:
            inp["b_up"] = rng.standard_normal((E, dff)) * 0.3
            inp["b_down"] = rng.standard_normal((E, d)) * 0.3
        if n_shared:
            inp["ws_up"] = rng.standard_normal((n_shared, dff, d)) * 0.5
            inp["ws_down"] = rng.standard_normal((n_shared, d, dff)) * 0.5
            if act == "swiglu":
                inp["ws_gate"] = rng.standard_normal((n_shared, dff, d)) * 0.5
        z = inp["x"] @ inp["w_router"].T
        if k == E or np.min(O.topk_gap(z, k)) > 0.05:
            return inp


def check_backward(o, b=None):
    """Finite differences of L = <dy, y> + dlb lb + dzl zl (forward oracle) against the analytic
    gradients, for every tensor; k = E with identical experts leaves the router only the losses."""
    if b is None:
        from oracle import moe_backward as b
    rng = np.random.default_rng(99)
    cases = [dict(T=7, d=5, E=4, k=2, dff=3, act="gelu", bias=True, n_shared=0, cf=0.75, tau=1.0),
             dict(T=6, d=4, E=3, k=2, dff=3, act="swiglu", bias=False, n_shared=1, cf=0.0, tau=1.0),
             dict(T=5, d=4, E=4, k=1, dff=2, act="swiglu", bias=False, n_shared=0, cf=1.0, tau=1.0),
             # router temperatures: the logits' gradient through z / tau
             dict(T=6, d=4, E=4, k=2, dff=3, act="gelu", bias=True, n_shared=1, cf=0.0, tau=0.6),
             dict(T=6, d=4, E=3, k=2, dff=2, act="swiglu", bias=False, n_shared=0, cf=0.9, tau=2.5)]
    for c in cases:
        cf = c.pop("cf")
        tau = c.pop("tau")
        inp = _bwd_case(rng, **c)
        kw = dict(E=c["E"], k=c["k"], act=c["act"], n_shared=c["n_shared"], cf=cf, lb_coef=0.3, z_coef=0.2,
                  dlb=1.0, dzl=1.0, temperature=tau)
        dy = rng.standard_normal((c["T"], c["d"]))
        g = b.moe_layer_backward(inp, dy, **kw)
        names = {"x": "dx", "w_router": "dw_router", "w_up": "dw_up", "w_down": "dw_down"}
        if c["act"] == "swiglu":
            names["w_gate"] = "dw_gate"
        if c["bias"]:
            names.update(b_up="db_up", b_down="db_down")
        if c["n_shared"]:
            names.update(ws_up="dws_up", ws_down="dws_down")
            if c["act"] == "swiglu":
                names["ws_gate"] = "dws_gate"
        h = 1e-6
        for tname, gname in names.items():
            assert g[gname].shape == inp[tname].shape, (gname, g[gname].shape)
            flat = inp[tname].reshape(-1)
            for i in rng.choice(flat.size, size=min(8, flat.size), replace=False):
                old = flat[i]
                flat[i] = old + h
                lp = b.objective(inp, dy, **kw)
                flat[i] = old - h
                lm = b.objective(inp, dy, **kw)
                flat[i] = old
                fd = (lp - lm) / (2 * h)
                an = g[gname].reshape(-1)[i]
                assert abs(an - fd) <= 1e-6 * (1.0 + abs(fd)), (c["act"], tname, int(i), an, fd)
    # k = E, identical experts: y = FFN(x) whatever the routing, so without the losses the router
    # gets no gradient, and with only the z-loss it gets 2 beta lse_t P_t / T through x
    inp = _bwd_case(rng, 6, 4, 3, 3, 3, "gelu", False, 0)
    for key in ("w_up", "w_down"):
        inp[key] = np.repeat(inp[key][:1], 3, axis=0)
    dy = rng.standard_normal((6, 4))
    g = b.moe_layer_backward(inp, dy, E=3, k=3, act="gelu", dlb=0.0, dzl=0.0)
    assert np.abs(g["dw_router"]).max() < 1e-12
    g = b.moe_layer_backward(inp, np.zeros((6, 4)), E=3, k=3, act="gelu", z_coef=0.5, dlb=0.0, dzl=1.0)
    P, lse = o.softmax_lse(inp["x"] @ inp["w_router"].T)
    np.testing.assert_allclose(g["dw_router"], ((2 * 0.5 * lse / 6)[:, None] * P).T @ inp["x"], rtol=1e-12, atol=1e-14)
    # the task loss <dy, y> is a sum over tokens, and dropless routing treats each token alone: its
    # gradient over a batch is the sum of the gradients over any split of the batch (what a data-
    # parallel all-reduce of per-rank gradients relies on); dx is the halves' rows side by side
    inp = _bwd_case(rng, 10, 5, 4, 2, 3, "swiglu", False, 1)
    dy = rng.standard_normal((10, 5))
    kw = dict(E=4, k=2, act="swiglu", n_shared=1, dlb=0.0, dzl=0.0)
    whole = b.moe_layer_backward(inp, dy, **kw)
    halves = []
    for sl in (slice(0, 4), slice(4, 10)):
        part = dict(inp)
        part["x"] = inp["x"][sl]
        halves.append(b.moe_layer_backward(part, dy[sl], **kw))
    for name, v in whole.items():
        if name == "dx":
            np.testing.assert_allclose(np.concatenate([halves[0]["dx"], halves[1]["dx"]]), v, rtol=1e-12, atol=1e-12)
        else:
            np.testing.assert_allclose(halves[0][name] + halves[1][name], v, rtol=1e-12, atol=1e-12, err_msg=name)


def check_fp8(o):
    # the definition against torch's float8_e4m3fn: every finite code decodes to the same value,
    # and encoding agrees on random in-range values (ties to even included)
    codes = torch.arange(256, dtype=torch.int64).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        v = o.e4m3_value(c)
        assert (math.isnan(v) and math.isnan(ref[c])) or v == ref[c], (c, v, ref[c])
    assert o.e4m3_value(0x7E) == 448.0 and o.e4m3_value(0x01) == 2.0 ** -9 and o.e4m3_value(0x38) == 1.0
    vals = np.concatenate([RNG.standard_normal(300) * 40, [1.0625, 1.1875, -3.3, 2.0 ** -10, 0.0, 447.0]])
    tq = torch.tensor(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, c in zip(vals, tq):
        assert o.e4m3_encode(v) == int(c) or (v == 0.0 and o.e4m3_value(o.e4m3_encode(v)) == 0.0), (v, c)
    assert o.e4m3_encode(1000.0) == 0x7E and o.e4m3_encode(-1000.0) == 0xFE   # saturating
    # per-row scaling: the row maximum maps to 448 exactly; relative error of normal values <= 2^-4
    W = RNG.standard_normal((5, 40)) * 0.02
    q = o.quantize_rows_e4m3(W)
    assert q["codes"].dtype == np.uint8 and q["scale"].dtype == np.float32
    amax = np.abs(W).max(axis=1)
    np.testing.assert_allclose(np.abs(q["dequantized"]).max(axis=1), amax, rtol=1e-6)
    normal = np.abs(W) / q["scale"].astype(np.float64)[:, None] >= 2.0 ** -6
    rel = np.abs(q["dequantized"] - W)[normal] / np.abs(W)[normal]
    assert rel.max() <= 2.0 ** -4 + 1e-7
    assert (o.quantize_rows_e4m3(np.zeros((2, 3)))["dequantized"] == 0).all()
    # the vectorised encoder agrees with the scalar definition, exact midpoints (ties) included
    tab = o.e4m3_table()
    mids = np.array([(tab[c] + tab[c + 1]) / 2 for c in range(0x7E)])
    vals = np.concatenate([RNG.standard_normal(600) * 40, RNG.standard_normal(200) * 0.01, mids, -mids,
                           [0.0, -0.0, 448.0, 449.0, 464.0, 1e9, -1e9, 2.0 ** -10, -3 * 2.0 ** -10]])
    arr = o.e4m3_encode_array(vals)
    assert arr.dtype == np.uint8
    assert all(int(a) == o.e4m3_encode(v) for a, v in zip(arr, vals))
    # float32 division (the rounding a float32 quantiser takes): codes equal torch's float32 quotient
    # converted by float8_e4m3fn, and the scale equals the float64 path's (one rounding either way)
    Wb = torch.tensor(RNG.standard_normal((40, 192)) * 0.02, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    Wb[3] = 0.0
    q32, q64 = o.quantize_rows_e4m3(Wb, "f32"), o.quantize_rows_e4m3(Wb)
    assert np.array_equal(q32["scale"], q64["scale"]) and q32["scale"][3] == 1.0
    t32 = torch.tensor(Wb, dtype=torch.float32) / torch.tensor(q32["scale"])[:, None]
    assert np.array_equal(t32.to(torch.float8_e4m3fn).view(torch.uint8).numpy(), q32["codes"])
    np.testing.assert_array_equal(o.dequantize_rows_e4m3(q32["codes"], q32["scale"]), q32["dequantized"])
    with pytest.raises(ValueError):
        o.quantize_rows_e4m3(Wb, "f16")


def check_int8(o):
    """INT8 per-row codes against brute force on exact rationals: the code is the integer of
    [-127, 127] nearest to the IEEE float32 quotient (torch's float32 division), ties to even;
    the row maximum maps to +-127; dequantised values lie within half a step of W."""
    rng = np.random.default_rng(21)
    W = torch.tensor(rng.standard_normal((12, 40)) * 0.02, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    W[5] = 0.0
    W[7, 3] = -np.abs(W[7]).max() * 1.5          # the row maximum on a negative entry
    q = o.quantize_rows_int8(W)
    assert q["codes"].dtype == np.int8 and q["scale"].dtype == np.float32
    W32 = torch.tensor(W, dtype=torch.float32)
    amax = W32.abs().amax(dim=1)
    scale = torch.where(amax > 0, amax / torch.tensor(127.0), torch.tensor(1.0))
    assert np.array_equal(scale.numpy(), q["scale"])
    quot = (W32 / scale[:, None]).numpy()
    for r in range(W.shape[0]):
        for c in range(W.shape[1]):
            x = Fraction(float(quot[r, c]))
            best = min(range(-127, 128), key=lambda n: (abs(x - n), n % 2))
            assert int(q["codes"][r, c]) == best, (r, c, float(x), best)
    assert q["scale"][5] == 1.0 and (q["codes"][5] == 0).all()
    for r in range(W.shape[0]):
        if r != 5:
            assert np.abs(q["codes"][r].astype(int)).max() == 127
    assert q["codes"][7, 3] == -127
    step = q["scale"].astype(np.float64)[:, None]
    assert (np.abs(q["dequantized"] - W) <= step / 2 * (1 + 1e-6)).all()
    # exact halves round to the even integer: rows scaled so that W / s = n + 1/2 exactly
    s = np.float32(2.0 ** -7)
    Wt = np.array([[127 * s, 0.5 * s, 1.5 * s, 2.5 * s, -2.5 * s, -0.5 * s, 126.5 * s]], np.float64)
    qt = o.quantize_rows_int8(Wt)
    assert qt["scale"][0] == s
    assert qt["codes"][0].tolist() == [127, 0, 2, 2, -2, 0, 126]
    # stacks of experts: separate rows, or one scale per row over blocks placed side by side
    Ws = rng.standard_normal((3, 4, 8)) * 0.02
    Ws[1, 2, 5] = 0.5
    sep = o.quantize_experts(Ws, "int8")
    assert sep["scale"].shape == (3, 4) and np.isclose(sep["scale"][1, 2], np.float32(0.5) / np.float32(127))
    joint = o.quantize_experts(Ws, "int8", joint_blocks=True)
    assert joint["scale"].shape == (4,) and joint["codes"].shape == (3, 4, 8)
    for r in range(4):
        assert joint["scale"][r] == np.float32(np.float32(np.abs(Ws[:, r, :]).max()) / np.float32(127))
    assert joint["codes"][1, 2, 5] == 127 and np.abs(joint["codes"][0, 2].astype(int)).max() < 127
    np.testing.assert_array_equal(joint["dequantized"][2], o.dequantize_rows_int8(joint["codes"][2], joint["scale"]))
    e = o.quantize_experts(Ws, "e4m3", joint_blocks=True)
    assert e["scale"][2] == np.float32(np.float32(0.5) / np.float32(448))


def check_routing_backward(b):
    """combine_backward and router_backward against torch autograd of the same composite: the
    combine y_t = sum_j w_tj y_perm[row_of[t, j]] (dropped slots excluded), and the router from x and
    W_r through z = x W_r^T, the renormalised softmax of the selected logits / tau, the load-balance
    loss with fixed counts and the z-loss."""
    rng = np.random.default_rng(51)
    T, d, E, k, tau = 7, 6, 5, 2, 1.7
    lb_coef, z_coef, dlb, dzl = 0.01, 0.001, 1.3, 0.7
    x = rng.standard_normal((T, d))
    Wr = rng.standard_normal((E, d))
    z = x @ Wr.T
    idx = O.topk_select(z, k)
    P, lse = O.softmax_lse(O.temper(z, tau))
    w = O.renormalise(P, idx)
    counts = np.bincount(idx.ravel(), minlength=E)
    dw = rng.standard_normal((T, k))
    rb = b.router_backward(x, Wr, P, lse, idx, w, dw, counts, E=E, k=k, lb_coef=lb_coef, z_coef=z_coef,
                           dlb=dlb, dzl=dzl, temperature=tau)
    xt = torch.tensor(x, requires_grad=True)
    wt = torch.tensor(Wr, requires_grad=True)
    zt = (xt @ wt.T) / tau
    sel = torch.gather(zt, 1, torch.tensor(idx))
    L = (torch.softmax(sel, dim=1) * torch.tensor(dw)).sum()
    Pt = torch.softmax(zt, dim=1)
    f = torch.tensor(counts / (T * k))
    L = L + dlb * lb_coef * E * (f * Pt.mean(dim=0)).sum()
    L = L + dzl * z_coef * (torch.logsumexp(zt, dim=1) ** 2).mean()
    L.backward()
    np.testing.assert_allclose(rb["dx"], xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(rb["dw_router"], wt.grad.numpy(), rtol=1e-10, atol=1e-12)
    # combine: a dropped slot (row -1) gets no gradient
    row_of = np.array([[0, 3], [1, -1], [2, 4], [5, 6], [7, -1], [8, 9], [10, 11]])
    y_perm = rng.standard_normal((12, d))
    dy = rng.standard_normal((T, d))
    cb = b.combine_backward(dy, y_perm, row_of, w)
    wv = torch.tensor(w, requires_grad=True)
    yv = torch.tensor(y_perm, requires_grad=True)
    y = torch.zeros((T, d), dtype=torch.float64)
    for t in range(T):
        for j in range(k):
            if row_of[t, j] >= 0:
                y[t] = y[t] + wv[t, j] * yv[row_of[t, j]]
    (y * torch.tensor(dy)).sum().backward()
    np.testing.assert_allclose(cb["dw"], wv.grad.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(cb["dy_perm"], yv.grad.numpy(), rtol=1e-12, atol=1e-14)


def check_backup_expert(o):
    """A backup expert identical to every routed expert makes drops invisible (the dropless layer);
    a zero backup expert gives the dropping layer; drops are counted."""
    rng = np.random.default_rng(11)
    T, d, E, k, f = 16, 5, 4, 2, 6
    W1, W2 = rng.standard_normal((f, d)), rng.standard_normal((d, f))
    b1, b2 = rng.standard_normal(f) * 0.1, rng.standard_normal(d) * 0.1
    inp = dict(x=rng.standard_normal((T, d)), w_router=rng.standard_normal((E, d)),
               w_up=np.repeat(W1[None], E, 0), w_down=np.repeat(W2[None], E, 0),
               b_up=np.repeat(b1[None], E, 0), b_down=np.repeat(b2[None], E, 0))
    same = dict(w_up=W1, w_down=W2, b_up=b1, b_down=b2)
    a = o.moe_layer_backup_expert(inp, same, E=E, k=k, act="gelu", cf=0.5)
    assert a["backup_rows"] > 0 and a["drops"] == a["backup_rows"]
    full = o.moe_layer(inp, E=E, k=k, act="gelu", cf=0.0)
    np.testing.assert_allclose(a["y"], full["y"], rtol=1e-12, atol=1e-12)
    # with identical experts and renormalised weights the output is the dense FFN itself
    np.testing.assert_allclose(a["y"], o.expert_ffn(inp["x"], "gelu", W1, W2, None, b1, b2), rtol=1e-12, atol=1e-12)
    zero = dict(w_up=np.zeros((f, d)), w_down=np.zeros((d, f)), b_up=np.zeros(f), b_down=np.zeros(d))
    b = o.moe_layer_backup_expert(inp, zero, E=E, k=k, act="gelu", cf=0.5)
    np.testing.assert_array_equal(b["y"], o.moe_layer(inp, E=E, k=k, act="gelu", cf=0.5)["y"])
    assert abs(a["lb"] - full["lb"]) < 1e-15 and abs(a["zl"] - full["zl"]) < 1e-15


def check_temperature(o):
    z = RNG.standard_normal((20, 6)) * 2
    assert np.array_equal(o.temper(z, 1.0), z)
    for tau in (0.5, 1.5, 4.0):
        zt = o.temper(z, tau)
        assert np.array_equal(o.topk_select(zt, 3), o.topk_select(z, 3))     # same experts chosen
        P, _ = o.softmax_lse(zt)
        idx = o.topk_select(zt, 2)
        w = o.renormalise(P, idx)
        # two selected experts: w_0 = sigmoid((z_a - z_b) / tau)
        za = np.take_along_axis(z, idx, axis=1)
        np.testing.assert_allclose(w[:, 0], sps.expit((za[:, 0] - za[:, 1]) / tau), rtol=1e-12)
    # a very hot router spreads its weights evenly; a cold one puts all weight on the top expert
    P, _ = o.softmax_lse(o.temper(z, 1e9))
    np.testing.assert_allclose(o.renormalise(P, o.topk_select(z, 3)), 1.0 / 3, rtol=1e-6)
    P, _ = o.softmax_lse(o.temper(z, 1e-6))
    w = o.renormalise(P, o.topk_select(z, 3))
    assert np.allclose(w[:, 0], 1.0) and np.allclose(w[:, 1:], 0.0)
    with pytest.raises(ValueError):
        o.temper(z, 0.0)
    # in the layer, tau acts on the logits before everything else: the same as a router (and logit
    # bias) divided by tau, whatever the drops and shared experts
    rng = np.random.default_rng(7)
    inp = _bwd_case(rng, 12, 5, 4, 2, 6, "swiglu", False, 1)
    inp["logit_bias"] = np.array([0.3, 0.0, -0.2, 0.1])
    for tau in (0.5, 3.0):
        a = o.moe_layer(inp, E=4, k=2, act="swiglu", n_shared=1, cf=0.8, temperature=tau)
        scaled = dict(inp, w_router=inp["w_router"] / tau, logit_bias=inp["logit_bias"] / tau)
        b = o.moe_layer(scaled, E=4, k=2, act="swiglu", n_shared=1, cf=0.8)
        assert np.array_equal(a["idx"], b["idx"]) and np.array_equal(a["row_of"], b["row_of"])
        np.testing.assert_allclose(a["y"], b["y"], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose([a["lb"], a["zl"]], [b["lb"], b["zl"]], rtol=1e-12)
        # and the losses differ from the untempered layer's (the temperature is not ignored)
        c = o.moe_layer(inp, E=4, k=2, act="swiglu", n_shared=1, cf=0.8)
        assert abs(c["zl"] - a["zl"]) > 1e-6


ALL_CHECKS = [check_router, check_softmax, check_topk, check_renormalise, check_capacity,
              check_dispatch, check_activations, check_expert_ffn, check_layer_reductions, check_combine_fixture,
              check_losses, check_coactivation, check_backward, check_fp8, check_int8, check_temperature,
              check_backup_expert]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(O)


def test_param_count_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "param_count_example.json")))
    M = 2 ** 20
    d, n, k = g["d_model"], g["n_expert"], g["top_k"]
    per = O.expert_param_count(d, g["d_ff_expert"], "gelu")
    assert round(per / M) == g["params_per_expert_M"]
    assert round(n * per / M) == g["params_all_experts_M"]
    assert round(O.expert_param_count(d, g["d_ff_dense"], "gelu") / M) == g["params_dense_ffn_M"]
    assert round(k * per / M) == g["params_active_M"]


def test_shape_contract_example():
    g = json.load(open(os.path.join(GOLDEN, "shape_contract_example.json")))
    T = g["batch_size"] * g["seq_len"]
    d, E, f, k = g["d_model"], g["num_experts"], g["expert_hidden_dim"], g["k"]
    rng = np.random.default_rng(7)
    inp = dict(x=rng.standard_normal((T, d)), w_router=rng.standard_normal((E, d)) * 0.02,
               w_up=rng.standard_normal((E, f, d)) * 0.02, w_down=rng.standard_normal((E, d, f)) * 0.02)
    out = O.moe_layer(inp, E=E, k=k, act="gelu")
    assert out["y"].reshape(g["batch_size"], g["seq_len"], d).shape == (g["batch_size"], g["seq_len"], d)


def test_flame_moe_config_matches_pages():
    from synth import WORKLOADS
    g = json.load(open(os.path.join(GOLDEN, "flame_moe_layer.json")))
    wl = WORKLOADS["finegrained_bf16"]
    assert wl.E == g["experts_per_layer"] and wl.n_shared == g["shared_experts"]
    assert wl.k == g["routed_top_k"] == g["active_per_token"] - g["shared_experts"]
    assert wl.lb_coef == g["load_balance_coef"] and wl.z_coef == g["router_z_loss_coef"]


# ----------------------------------------------------------------------------- planted mistakes
def _mut_router_transposed(x, w, b=None):
    z = np.asarray(x, np.float64) @ np.asarray(w, np.float64).T[::-1]
    return z


def _mut_topk_high_index(z, k):
    T, E = z.shape
    order = np.lexsort((-np.broadcast_to(np.arange(E), (T, E)), -z), axis=-1)
    return order[:, :k]


def _mut_no_renorm(P, idx):
    return np.take_along_axis(P, idx, axis=1)


_REAL = dict(dispatch=O.dispatch, aux_losses=O.aux_losses, expert_ffn=O.expert_ffn)


def _mut_dispatch_reverse(idx, E, cap):
    return _REAL["dispatch"](idx[::-1].copy(), E, cap)


def _mut_lb_without_E(P, lse, counts, k, a, b):
    lb, zl = _REAL["aux_losses"](P, lse, counts, k, a, b)
    return lb / P.shape[1] if P.shape[0] else lb, zl


def _mut_gelu_tanh(u):
    return 0.5 * u * (1 + np.tanh(math.sqrt(2 / math.pi) * (u + 0.044715 * u ** 3)))


def _mut_ffn_no_bias(xr, act, w_up, w_down, w_gate=None, b_up=None, b_down=None):
    return _REAL["expert_ffn"](xr, act, w_up, w_down, w_gate, b_up, None)


def _mut_capacity_floor(cf, T, k, E):
    return None if cf <= 0 else int(cf * T * k // E)


def _mut_combine_unweighted(idx, w, row_of, y_perm, tokens, y_shared=None):
    return O_combine(idx, np.ones_like(w), row_of, y_perm, tokens, y_shared)


def _mut_combine_reversed_slots(idx, w, row_of, y_perm, tokens, y_shared=None):
    # each slot's weight paired with the other slot's row (the weights reversed across the slots)
    return O_combine(idx, np.ascontiguousarray(w[:, ::-1]), row_of, y_perm, tokens, y_shared)


def _mut_silu_sigmoid(u):
    return sps.expit(u)


O_combine = O.combine


def _mut_e4m3_bias8(code):
    v = _REAL_E4M3(code)
    return v / 2.0 if v == v else v


_REAL_E4M3 = O.e4m3_value


def _mut_e4m3_ties_away(v):
    v = np.asarray(v, np.float64)
    vals = O.e4m3_table()[:0x7F]
    a = np.minimum(np.abs(v), 448.0)
    hi = np.minimum(np.searchsorted(vals, a, side="left"), 0x7E)
    lo = np.maximum(hi - 1, 0)
    code = np.where(a - vals[lo] < vals[hi] - a, lo, hi)
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def _mut_int8_ties_away(W):
    W32 = np.asarray(W, np.float64).astype(np.float32)
    amax = np.abs(W32).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(127.0), np.float32(1.0)).astype(np.float32)
    q = (W32 / scale[:, None]).astype(np.float64)
    codes = np.clip(np.sign(q) * np.floor(np.abs(q) + 0.5), -127, 127).astype(np.int8)
    return dict(codes=codes, scale=scale, dequantized=codes * scale.astype(np.float64)[:, None])


def _mut_int8_scale_128(W):
    W32 = np.asarray(W, np.float64).astype(np.float32)
    amax = np.abs(W32).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(128.0), np.float32(1.0)).astype(np.float32)
    codes = np.clip(np.rint(W32 / scale[:, None]), -127, 127).astype(np.int8)
    return dict(codes=codes, scale=scale, dequantized=codes * scale.astype(np.float64)[:, None])


_REAL_QUANT_EXPERTS = O.quantize_experts


def _mut_quant_experts_no_joint(W, fmt, joint_blocks=False):
    r = _REAL_QUANT_EXPERTS(W, fmt, False)
    if joint_blocks:
        r = dict(r, scale=r["scale"][0])
    return r


def _mut_coact_upper_only(idx, E):
    C = np.zeros((E, E), dtype=np.int64)
    for row in np.asarray(idx):
        for a in row:
            for b in row:
                if a <= b:
                    C[int(a), int(b)] += 1
    return C


@pytest.mark.parametrize("name,fn,check", [
    ("router_logits", _mut_router_transposed, check_router),
    ("topk_select", _mut_topk_high_index, check_topk),
    ("renormalise", _mut_no_renorm, check_renormalise),
    ("dispatch", _mut_dispatch_reverse, check_dispatch),
    ("aux_losses", _mut_lb_without_E, check_losses),
    ("gelu_erf", _mut_gelu_tanh, check_activations),
    ("expert_ffn", _mut_ffn_no_bias, check_expert_ffn),
    ("capacity", _mut_capacity_floor, check_capacity),
    ("combine", _mut_combine_unweighted, check_layer_reductions),
    ("combine", _mut_combine_unweighted, check_combine_fixture),
    ("combine", _mut_combine_reversed_slots, check_combine_fixture),
    ("silu", _mut_silu_sigmoid, check_expert_ffn),
    ("coactivation", _mut_coact_upper_only, check_coactivation),
    ("e4m3_value", _mut_e4m3_bias8, check_fp8),
    ("e4m3_encode_array", _mut_e4m3_ties_away, check_fp8),
    ("quantize_rows_int8", _mut_int8_ties_away, check_int8),
    ("quantize_rows_int8", _mut_int8_scale_128, check_int8),
    ("quantize_experts", _mut_quant_experts_no_joint, check_int8),
])
def test_planted_mistakes_are_caught(name, fn, check, monkeypatch):
    """Plant one mistake in the oracle module itself (so its internal callers see it too)."""
    real = getattr(O, name)
    monkeypatch.setattr(O, name, fn)
    with pytest.raises((AssertionError, ValueError, IndexError)):
        check(O)
    monkeypatch.setattr(O, name, real)


# planted mistakes in the backward oracle (patched in oracle.moe_backward itself)
def _mut_gelu_grad_no_density(u):
    return 0.5 * (1.0 + sps.erf(np.asarray(u) / math.sqrt(2.0)))


def _mut_silu_grad_sigmoid(u):
    return sps.expit(u)


@pytest.mark.parametrize("name,fn", [
    ("gelu_erf_grad", _mut_gelu_grad_no_density),
    ("silu_grad", _mut_silu_grad_sigmoid),
    ("expert_ffn_backward", "dx_halved"),
])
def test_planted_backward_mistakes_are_caught(name, fn, monkeypatch):
    from oracle import moe_backward as B
    real = getattr(B, name)
    if fn == "dx_halved":
        def fn(*a, **kw):
            out = dict(real(*a, **kw))
            out["dx"] = 0.5 * out["dx"]
            return out
    monkeypatch.setattr(B, name, fn)
    with pytest.raises(AssertionError):
        check_backward(O, B)



def test_routing_backward_pin():
    from oracle import moe_backward as B
    check_routing_backward(B)


@pytest.mark.parametrize("name,mistake", [
    ("router_backward", "no_temperature"),
    ("router_backward", "z_loss_dropped"),
    ("combine_backward", "row_scale_wrong"),
])
def test_planted_routing_backward_mistakes_are_caught(name, mistake, monkeypatch):
    from oracle import moe_backward as B
    real = getattr(B, name)

    def fn(*a, **kw):
        if mistake == "no_temperature":
            kw = dict(kw, temperature=1.0)
        if mistake == "z_loss_dropped":
            kw = dict(kw, dzl=0.0)
        out = dict(real(*a, **kw))
        if mistake == "row_scale_wrong":
            out["dy_perm"] = np.where(out["dy_perm"] != 0, out["dy_perm"] * 1.5, 0.0)
        return out
    monkeypatch.setattr(B, name, fn)
    with pytest.raises(AssertionError):
        check_routing_backward(B)
