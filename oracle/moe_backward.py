"""CPU oracle of the backward pass of the sparse MoE FFN layer (the first of the later rows: the
pages train these layers with the load-balance and z-loss terms added to the objective).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests may import this module.  It shares no code
with the CUDA library.

The gradients are the chain rule through the forward definition in moe_oracle.py, in float64,
with an explicit loop over experts.  The objective is

    L = sum_t <dy_t, y_t> + dlb * lb + dzl * zl

for an upstream gradient dy [T, d] and weights dlb, dzl of the two auxiliary losses (the router
z-loss coefficient of the FLAME-MoE summary, sec. 2; the load-balance loss of the OpenMythos
article, sec. 3.1).  Top-k selection and capacity drops are piecewise constant in the logits, so
they pass no gradient; the expert fractions f_e = counts_e / (T k) of the load-balance loss are
counts and pass none either, which leaves its gradient on the mean probabilities P_e.

Pins (tests/test_oracle_pins.py, check_backward): central finite differences of L, computed with
the pinned forward oracle, on small layers whose top-k margins are far larger than the step, for
every parameter tensor and the input; k = E with identical experts, where the output does not
depend on the router, so the router's gradient is exactly that of the two losses; and the task
loss's gradients over a dropless batch equal the sums of those over any split of it.  The routing
half also against torch autograd (check_routing_backward).
"""
from __future__ import annotations

import math
from typing import Dict

import numpy as np
from scipy import special as _sp

from . import moe_oracle as O


def gelu_erf_grad(u: np.ndarray) -> np.ndarray:
    """d/du of u Phi(u) = Phi(u) + u phi(u)."""
    u = np.asarray(u, np.float64)
    return 0.5 * (1.0 + _sp.erf(u / math.sqrt(2.0))) + u * np.exp(-0.5 * u * u) / math.sqrt(2.0 * math.pi)


def silu_grad(u: np.ndarray) -> np.ndarray:
    """d/du of u sigmoid(u) = sigmoid(u) (1 + u (1 - sigmoid(u)))."""
    s = _sp.expit(np.asarray(u, np.float64))
    return s * (1.0 + u * (1.0 - s))


def expert_ffn_backward(xr, act: str, dY, w_up, w_down, w_gate=None, b_up=None) -> Dict[str, np.ndarray]:
    """Gradients of sum <dY, FFN(xr)> for one expert (rows xr [n, d], nn.Linear weights [out, in]):
    dx [n, d], dw_up, dw_down, dw_gate (SwiGLU), db_up and db_down (GELU with biases)."""
    xr = np.asarray(xr, np.float64)
    dY = np.asarray(dY, np.float64)
    W1 = np.asarray(w_up, np.float64)
    W2 = np.asarray(w_down, np.float64)
    out: Dict[str, np.ndarray] = {}
    if act == "gelu":
        a = xr @ W1.T
        if b_up is not None:
            a = a + np.asarray(b_up, np.float64)[None, :]
        h = O.gelu_erf(a)
        out["dw_down"] = dY.T @ h
        out["db_down"] = dY.sum(axis=0)
        da = (dY @ W2) * gelu_erf_grad(a)
        out["dw_up"] = da.T @ xr
        out["db_up"] = da.sum(axis=0)
        out["dx"] = da @ W1
    elif act == "swiglu":
        Wg = np.asarray(w_gate, np.float64)
        g = xr @ Wg.T
        u = xr @ W1.T
        h = O.silu(g) * u
        out["dw_down"] = dY.T @ h
        dh = dY @ W2
        du = dh * O.silu(g)
        dg = dh * u * silu_grad(g)
        out["dw_up"] = du.T @ xr
        out["dw_gate"] = dg.T @ xr
        out["dx"] = du @ W1 + dg @ Wg
    else:
        raise ValueError(act)
    return out


def combine_backward(dy, y_perm, row_of, w) -> Dict[str, np.ndarray]:
    """Backward of the combine y_t = sum over kept slots j of w_tj y_perm[row_of[t, j]] (+ shared):
    dw [T, k] = <dy_t, y_perm[row]> (0 for a dropped slot) and dy_perm [rows, d], the upstream
    gradient of each kept row, w_tj dy_t."""
    dy = np.asarray(dy, np.float64)
    y_perm = np.asarray(y_perm, np.float64)
    row_of = np.asarray(row_of)
    T, k = row_of.shape
    dw = np.zeros((T, k))
    dy_perm = np.zeros_like(y_perm)
    for t in range(T):
        for j in range(k):
            r = int(row_of[t, j])
            if r >= 0:
                dw[t, j] = float(dy[t] @ y_perm[r])
                dy_perm[r] = w[t, j] * dy[t]
    return dict(dw=dw, dy_perm=dy_perm)


def router_backward(x, w_router, P, lse, idx, w, dw, counts, *, E: int, k: int, lb_coef: float = 0.01,
                    z_coef: float = 0.001, dlb: float = 1.0, dzl: float = 1.0,
                    temperature: float = 1.0) -> Dict[str, np.ndarray]:
    """Backward of the router given dL/dw_tj (dw [T, k]) and the weights of the two losses:
    the renormalised top-k weights are a softmax over the k selected logits, so
    dz_e = w_e (dw_e - sum_i w_i dw_i) for the selected e (top-k selection itself passes no
    gradient); the load-balance loss alpha E sum_e f_e Pbar_e adds, through the full softmax,
    P_te (g_e - sum_e' P_te' g_e') with g_e = dlb alpha E f_e / T (f_e = counts_e / (T k), counts
    pass no gradient); the z-loss beta mean_t lse_t^2 adds dzl 2 beta lse_t P_te / T; a router
    temperature divides the whole by tau.  Returns dz [T, E], dw_router = dz^T x [E, d] and
    dx = dz W_r [T, d]."""
    x = np.asarray(x, np.float64)
    Wr = np.asarray(w_router, np.float64)
    P = np.asarray(P, np.float64)
    T = x.shape[0]
    dz = np.zeros((T, E))
    for t in range(T):
        s = float(w[t] @ dw[t])
        for j in range(k):
            dz[t, int(idx[t, j])] += w[t, j] * (dw[t, j] - s)
    if T > 0:
        f = np.asarray(counts, np.float64) / float(T * k)
        gP = dlb * lb_coef * E * f / T
        dz += P * (gP[None, :] - (P @ gP)[:, None])
        dz += (dzl * 2.0 * z_coef * np.asarray(lse, np.float64) / T)[:, None] * P
    dz = dz / float(temperature)
    return dict(dz=dz, dw_router=dz.T @ x, dx=dz @ Wr)


def moe_layer_backward(inp: Dict, dy, *, E: int, k: int, act: str, n_shared: int = 0, cf: float = 0.0,
                       lb_coef: float = 0.01, z_coef: float = 0.001, dlb: float = 1.0,
                       dzl: float = 1.0, temperature: float = 1.0) -> Dict[str, np.ndarray]:
    """Gradients of L = sum_t <dy_t, y_t> + dlb lb + dzl zl with respect to x, the router weights,
    every routed expert's weights (stacked [E, ...]) and every shared expert's (stacked [S, ...]).
    With a router temperature tau the layer sees z / tau, so the logits' gradient is divided by tau."""
    fwd = O.moe_layer(inp, E=E, k=k, act=act, n_shared=n_shared, cf=cf, lb_coef=lb_coef, z_coef=z_coef,
                      temperature=temperature)
    x = np.asarray(inp["x"], np.float64)
    dy = np.asarray(dy, np.float64)
    T, d = x.shape
    Wr = np.asarray(inp["w_router"], np.float64)
    P, lse, idx, w = fwd["P"], fwd["lse"], fwd["idx"], fwd["w"]
    row_of, tok_of, y_perm = fwd["row_of"], fwd["tok_of"], fwd["y_perm"]

    # combine: y_t = sum over kept slots of w_tj F_tj  ->  dL/dw_tj = <dy_t, F_tj>, 0 if dropped
    cb = combine_backward(dy, y_perm, row_of, w)
    dw = cb["dw"]
    slot_of_row = {}
    for t in range(T):
        for j in range(k):
            r = int(row_of[t, j])
            if r >= 0:
                slot_of_row[r] = (t, j)
    rb = router_backward(x, Wr, P, lse, idx, w, dw, fwd["counts"], E=E, k=k, lb_coef=lb_coef, z_coef=z_coef,
                         dlb=dlb, dzl=dzl, temperature=temperature)
    g: Dict[str, np.ndarray] = {"dw_router": rb["dw_router"], "dx": rb["dx"].copy()}

    # routed experts: row r of expert e carries w_tj dy_t
    has_bias = inp.get("b_up") is not None
    shapes = dict(dw_up=np.shape(inp["w_up"]), dw_down=np.shape(inp["w_down"]))
    if act == "swiglu":
        shapes["dw_gate"] = np.shape(inp["w_gate"])
    if has_bias:
        shapes["db_up"] = np.shape(inp["b_up"])
        shapes["db_down"] = np.shape(inp["b_down"])
    for name, shp in shapes.items():
        g[name] = np.zeros(shp)
    offsets = fwd["offsets"]
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi <= lo:
            continue
        rows = list(range(lo, hi))
        toks = tok_of[rows]
        wt = np.array([w[slot_of_row[r]] for r in rows])
        ge = expert_ffn_backward(x[toks], act, wt[:, None] * dy[toks], inp["w_up"][e], inp["w_down"][e],
                                 None if act != "swiglu" else inp["w_gate"][e],
                                 inp["b_up"][e] if has_bias else None)
        for name in shapes:
            g[name][e] += ge[name]
        np.add.at(g["dx"], toks, ge["dx"])

    # shared experts: weight 1 on every token
    if n_shared > 0:
        g["dws_up"] = np.zeros(np.shape(inp["ws_up"]))
        g["dws_down"] = np.zeros(np.shape(inp["ws_down"]))
        if act == "swiglu":
            g["dws_gate"] = np.zeros(np.shape(inp["ws_gate"]))
        for s_ in range(n_shared):
            gs = expert_ffn_backward(x, act, dy, inp["ws_up"][s_], inp["ws_down"][s_],
                                     None if act != "swiglu" else inp["ws_gate"][s_])
            g["dws_up"][s_] += gs["dw_up"]
            g["dws_down"][s_] += gs["dw_down"]
            if act == "swiglu":
                g["dws_gate"][s_] += gs["dw_gate"]
            g["dx"] += gs["dx"]
    return g


def objective(inp: Dict, dy, *, E: int, k: int, act: str, n_shared: int = 0, cf: float = 0.0,
              lb_coef: float = 0.01, z_coef: float = 0.001, dlb: float = 1.0, dzl: float = 1.0,
              temperature: float = 1.0) -> float:
    """L = sum_t <dy_t, y_t> + dlb lb + dzl zl from the forward oracle (for finite differences)."""
    fwd = O.moe_layer(inp, E=E, k=k, act=act, n_shared=n_shared, cf=cf, lb_coef=lb_coef, z_coef=z_coef,
                      temperature=temperature)
    return float(np.sum(np.asarray(dy, np.float64) * fwd["y"])) + dlb * fwd["lb"] + dzl * fwd["zl"]
