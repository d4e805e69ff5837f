"""CPU oracle of the forward pass of one sparse Mixture-of-Experts FFN layer.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import this module.  It shares no code with the CUDA library
and the library never calls it.

Everything is computed in float64 from the exact (bf16 or fp32) tensors the GPU consumes,
with an explicit loop over experts, in the order the sources describe the layer:

  1. router logits  z = x W_r^T (+ a fixed logit bias)      -- mini-moe tutorial, sec. 3.1
     (MoELayer: the router is a bias-free Linear); GPT-4 2%-parameters article, sec. 3.2
  2. P = softmax(z) per token, lse = logsumexp(z)            -- mini-moe tutorial, sec. 3.1
  3. top-k experts by descending logit                       -- mini-moe tutorial, sec. 3.1
     (torch.topk); the pages fix no tie rule, so equal logits go to the lower expert index
  4. weights renormalised over the k selected, w = P_sel / sum P_sel
                                                              -- mini-moe tutorial, sec. 3.1;
     OpenMythos article, sec. 3.1 (routing pseudo-code); equal to the GPT-4 article's softmax
     over the k selected logits (sec. 4.1 MoELayer)
  5. capacity C = ceil(cf * T * k / E) (exact rational ceil), assignments of each expert ranked in
     token order, rank >= C dropped (weight 0, no renormalisation)
                                                              -- OpenMythos article, sec. 3.1
     (capacity factor and overflow handling)
  6. expert FFN: GELU(erf) form  W2 gelu(W1 x + b1) + b2      -- mini-moe tutorial, sec. 3.1
                 SwiGLU form     Wd (silu(Wg x) * (Wu x))     -- GPT-4 article, sec. 3.1
  7. y_t = sum over kept slots of w_tj FFN_{e_tj}(x_t) + sum over shared experts FFN_s(x_t)
                                                              -- FLAME-MoE summary, sec. 2
     (weighted sum of the selected experts; 2 shared experts active for every token)
  8. load-balance loss  lb = alpha * E * sum_e f_e * Pbar_e, f_e = counts_e / (T k),
     Pbar_e = mean_t P_te                                     -- OpenMythos article, sec. 3.1
     router z-loss      zl = beta * mean_t lse_t^2            -- named but not written out in the
     FLAME-MoE summary, sec. 2; the formula used is the standard router z-loss

Pins (tests/test_oracle_pins.py): each function here is checked against something other than
itself -- brute-force sorting, closed forms, library routines (torch.nn.functional) on special
cases that reduce to a dense FFN, and hand-worked fixtures under tests/golden/.  The numeric
value of a full layer on random inputs has no worked example on the pages: beyond those
reductions it is "parity unpinned" by the pages and rests on the pinned parts.
"""
from __future__ import annotations

import math
from fractions import Fraction
from typing import Dict, Optional, Sequence

import numpy as np
from scipy import special as _sp


def _f64(a) -> Optional[np.ndarray]:
    """Widen a torch tensor or array-like to a float64 numpy array (exact for bf16/fp32)."""
    if a is None:
        return None
    if hasattr(a, "detach"):
        import torch  # local: only for the dtype conversion
        return a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


# ----------------------------------------------------------------------------- routing
def router_logits(x, w_router, logit_bias=None) -> np.ndarray:
    """z[t, e] = sum_i x[t, i] W_r[e, i] (+ logit_bias[e]).

    mini-moe tutorial, sec. 3.1: the router is one Linear(hidden_dim -> num_experts) without
    bias; the optional fixed bias vector models the skewed-routing workload (routing collapse,
    Naive-N0.5-Flash article sec. 2.2)."""
    z = _f64(x) @ _f64(w_router).T
    if logit_bias is not None:
        z = z + _f64(logit_bias)[None, :]
    return z


def temper(z: np.ndarray, temperature: float = 1.0) -> np.ndarray:
    """Router temperature (a routing variant): the logits divided by tau before the softmax, the
    top-k and the losses, as the GPT-4 2%-parameters article's routing-collapse tips describe
    (tau = 1 by default; a larger tau flattens the distribution).  The top-k choice is unchanged
    for tau > 0; the renormalised weights become a softmax of z_selected / tau."""
    if not temperature > 0:
        raise ValueError("temperature must be positive")
    return np.asarray(z, np.float64) / float(temperature)


def softmax_lse(z: np.ndarray):
    """Row softmax P and log-sum-exp lse of the logits (max-subtracted)."""
    if z.shape[0] == 0:
        return np.zeros_like(z), np.zeros(0)
    m = z.max(axis=1, keepdims=True)
    ex = np.exp(z - m)
    s = ex.sum(axis=1, keepdims=True)
    return ex / s, (m + np.log(s))[:, 0]


def topk_select(z: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits per token, in descending order; equal logits are ordered
    by ascending expert index (so the lower index wins a tie at the k-th place)."""
    T, E = z.shape
    if T == 0:
        return np.zeros((0, k), dtype=np.int64)
    order = np.lexsort((np.broadcast_to(np.arange(E), (T, E)), -z), axis=-1)
    return order[:, :k].astype(np.int64)


def topk_gap(z: np.ndarray, k: int) -> np.ndarray:
    """z_(k) - z_(k+1): the logit margin at the selection boundary (+inf when k == E)."""
    T, E = z.shape
    if k >= E:
        return np.full(T, np.inf)
    zs = -np.sort(-z, axis=1)
    return zs[:, k - 1] - zs[:, k]


def renormalise(P: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """w_tj = P[t, idx_tj] / sum_j P[t, idx_tj]."""
    sel = np.take_along_axis(P, idx, axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


# ----------------------------------------------------------------------------- dispatch
def capacity(cf: float, T: int, k: int, E: int) -> Optional[int]:
    """Expert capacity ceil(cf * T * k / E), exact in rationals (cf taken as the float32 value
    the C struct carries); None when cf <= 0 (dropless)."""
    if cf <= 0:
        return None
    cf32 = float(np.float32(cf))
    return int(math.ceil(Fraction(cf32) * T * k / E))


def dispatch(idx: np.ndarray, E: int, cap: Optional[int]) -> Dict[str, np.ndarray]:
    """Expert-sorted layout of the routed (token, slot) assignments.

    Each expert's assignments are ranked in increasing token order; rank >= cap is dropped.
    Kept rows are laid out expert after expert, tokens ascending inside an expert."""
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    rank = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            rank[t, j] = counts[e]
            counts[e] += 1
    kept_counts = counts.copy() if cap is None else np.minimum(counts, cap)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(kept_counts)
    row_of = np.full((T, k), -1, dtype=np.int64)
    tok_of = np.zeros(int(offsets[E]), dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            if cap is None or rank[t, j] < cap:
                r = int(offsets[e] + rank[t, j])
                row_of[t, j] = r
                tok_of[r] = t
    return dict(counts=counts, kept_counts=kept_counts, offsets=offsets, row_of=row_of,
                tok_of=tok_of, drops=int(T * k - offsets[E]))


# ----------------------------------------------------------------------------- experts
def gelu_erf(u: np.ndarray) -> np.ndarray:
    """GELU in its exact erf form, u * (1 + erf(u / sqrt 2)) / 2 (torch's nn.GELU default)."""
    return 0.5 * u * (1.0 + _sp.erf(u / math.sqrt(2.0)))


def silu(u: np.ndarray) -> np.ndarray:
    """SiLU u * sigmoid(u)."""
    return u * _sp.expit(u)


def expert_ffn(xr, act: str, w_up, w_down, w_gate=None, b_up=None, b_down=None) -> np.ndarray:
    """One expert on rows xr [n, d]; weights in nn.Linear layout [out, in].

    gelu:   W_down gelu(W_up x + b_up) + b_down   (mini-moe tutorial, sec. 3.1 experts)
    swiglu: W_down (silu(W_gate x) * (W_up x))     (GPT-4 article, sec. 3.1)"""
    xr = _f64(xr)
    if act == "gelu":
        u = xr @ _f64(w_up).T
        if b_up is not None:
            u = u + _f64(b_up)[None, :]
        h = gelu_erf(u)
    elif act == "swiglu":
        h = silu(xr @ _f64(w_gate).T) * (xr @ _f64(w_up).T)
    else:
        raise ValueError(act)
    y = h @ _f64(w_down).T
    if b_down is not None:
        y = y + _f64(b_down)[None, :]
    return y


def combine(idx, w, row_of, y_perm, tokens: Sequence[int], y_shared=None) -> np.ndarray:
    """y_t = sum over kept slots j (row_of >= 0) of w_tj * y_perm[row_of_tj]  (+ shared output)."""
    d = y_perm.shape[1] if y_perm.ndim == 2 and y_perm.shape[0] else (
        y_shared.shape[1] if y_shared is not None else 0)
    y = np.zeros((len(tokens), d))
    for i, t in enumerate(tokens):
        for j in range(idx.shape[1]):
            r = row_of[t, j]
            if r >= 0:
                y[i] += w[t, j] * y_perm[r]
        if y_shared is not None:
            y[i] += y_shared[i]
    return y


# ----------------------------------------------------------------------------- losses
def aux_losses(P: np.ndarray, lse: np.ndarray, counts: np.ndarray, k: int,
               lb_coef: float, z_coef: float):
    """(load-balance loss, router z-loss).  lb = alpha E sum_e f_e Pbar_e with f_e = counts_e/(T k)
    (pre-drop router counts) and Pbar_e = mean_t P_te; zl = beta mean_t lse_t^2.  Both are 0 for
    an empty batch."""
    T, E = P.shape
    if T == 0:
        return 0.0, 0.0
    f = counts / float(T * k)
    pbar = P.sum(axis=0) / T
    lb = lb_coef * E * float(np.sum(f * pbar))
    zl = z_coef * float(np.sum(lse * lse)) / T
    return lb, zl


def lb_loss_squared_mean_form(P: np.ndarray, lb_coef: float) -> float:
    """Diagnostic variant from the mini-moe tutorial, sec. 3.1 (its auxiliary loss): alpha E sum_e Pbar_e^2."""
    E = P.shape[1]
    pbar = P.mean(axis=0)
    return lb_coef * E * float(np.sum(pbar * pbar))


def lb_loss_kl_frequency_form(P: np.ndarray, counts: np.ndarray, lb_coef: float, eps: float = 1e-8) -> float:
    """Variant from the GPT-4 2%-parameters article, sec. 4.2 (its load-balancing loss): alpha times
    the KL divergence of the mean router probabilities Pbar from the uniform distribution,
    sum_e (1/E)(ln(1/E) - ln(Pbar_e + eps)), plus the squared distance of the selection frequencies
    f_e = counts_e / sum counts from 1/E.  eps is the article's smoothing inside the logarithm."""
    P = np.asarray(P, np.float64)
    E = P.shape[1]
    pbar = P.mean(axis=0)
    u = 1.0 / E
    kl = float(np.sum(u * (math.log(u) - np.log(pbar + eps))))
    c = np.asarray(counts, np.float64)
    f = c / c.sum() if c.sum() > 0 else np.zeros(E)
    return lb_coef * (kl + float(np.sum((f - u) ** 2)))


def moe_layer_backup_expert(inp: Dict, backup: Dict, *, E: int, k: int, act: str, n_shared: int = 0,
                             cf: float = 0.0, lb_coef: float = 0.01, z_coef: float = 0.001) -> Dict:
    """Routing variant with a backup expert: the mini-moe tutorial, sec. 6, says that tokens over an
    expert's capacity are dropped or routed to a backup expert.  Here every assignment the capacity
    drops goes to one extra expert (weights in ``backup``: w_up, w_down, and w_gate / b_up / b_down
    as the layer's experts have them), keeping its routing weight:
        y_t = (the layer's y_t) + sum over dropped slots j of w_tj FFN_backup(x_t).
    Routing, counts and both losses are the layer's own."""
    out = moe_layer(inp, E=E, k=k, act=act, n_shared=n_shared, cf=cf, lb_coef=lb_coef, z_coef=z_coef)
    x = _f64(inp["x"])
    T = x.shape[0]
    y = out["y"].copy()
    for t in range(T):
        for j in range(k):
            if int(out["row_of"][t, j]) < 0:
                f = expert_ffn(x[t:t + 1], act, backup["w_up"], backup["w_down"], backup.get("w_gate"),
                               backup.get("b_up"), backup.get("b_down"))
                y[t] += out["w"][t, j] * f[0]
    return dict(out, y=y, backup_rows=int(np.sum(np.asarray(out["row_of"]) < 0)))


def expert_param_count(d: int, dff: int, act: str = "gelu", bias: bool = False) -> int:
    """Weights of one expert: 2 d dff for the two-matrix form (Naive-N0.5-Flash article sec. 3.3),
    3 d dff for SwiGLU; biases add dff + d."""
    n = (3 if act == "swiglu" else 2) * d * dff
    return n + ((dff + d) if bias else 0)


# ----------------------------------------------------------------------------- routing statistics
def coactivation(idx: np.ndarray, E: int) -> np.ndarray:
    """Expert co-activation counts.  C[i, j] (i != j) = number of tokens whose selected experts
    include both i and j; C[i, i] = number of tokens that chose i.  The FLAME-MoE summary's
    directed co-activation score from E_i to E_j (expert co-activation analysis, fig. 5) is the
    conditional probability C[i, j] / C[i, i].  Plain loop over the tokens and their slot pairs."""
    C = np.zeros((E, E), dtype=np.int64)
    for row in np.asarray(idx):
        for a in row:
            for b in row:
                C[int(a), int(b)] += 1
    return C


def coactivation_score(C: np.ndarray) -> np.ndarray:
    """Directed score S[i, j] = P(j chosen | i chosen) = C[i, j] / C[i, i] (0 for unused i)."""
    d = np.diag(C).astype(np.float64)
    with np.errstate(invalid="ignore", divide="ignore"):
        S = np.where(d[:, None] > 0, C / d[:, None], 0.0)
    return S


def router_entropy(z: np.ndarray) -> float:
    """Mean over tokens of the entropy of the router distribution, -sum_e P_te ln P_te (nats), from
    the logits: H_t = lse_t - sum_e P_te z_te.  A low value means confident (or collapsed) routing,
    ln E a uniform one -- the routing-collapse signal the GPT-4 2% article's tips watch."""
    z = np.asarray(z, np.float64)
    if z.shape[0] == 0:
        return 0.0
    P, lse = softmax_lse(z)
    return float(np.mean(lse - np.sum(P * z, axis=1)))


def routing_stats(idx: np.ndarray, E: int, k: int, offsets=None):
    """(load imbalance, dropped fraction).  Imbalance: the busiest expert's token count over the
    uniform share T k / E that the load-balance loss of the OpenMythos article, sec. 3.1, pushes
    towards (1 = uniform).  Dropped fraction: assignments past the capacity (same section) over
    all T k, from offsets[E] = kept assignments; 0 without offsets."""
    idx = np.asarray(idx)
    tk = int(idx.shape[0]) * k
    if tk == 0:
        return 0.0, 0.0
    counts = np.bincount(idx.ravel(), minlength=E)
    dropped = 0.0 if offsets is None else (tk - int(offsets[E])) / tk
    return float(counts.max()) * E / tk, dropped


# ----------------------------------------------------------------------------- FP8 expert weights
# Weight-only FP8 experts (a later row: the decode-shaped layer is bound by reading its expert
# weights, so storing them in one byte halves the bytes).  Codes are OCP FP8 E4M3 ("fn": sign, 4
# exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite
# 448), one fp32 scale per output row (nn.Linear row) = max |w| / 448.

def e4m3_value(code: int) -> float:
    """Value of an E4M3 code by its definition (NaN for S.1111.111)."""
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_encode(v: float) -> int:
    """Nearest E4M3 code (ties to the even mantissa), saturating at +-448."""
    v = float(v)
    if math.isnan(v):
        raise ValueError("NaN has no E4M3 encoding here")
    sign = 0x80 if (v < 0 or (v == 0 and math.copysign(1.0, v) < 0)) else 0
    a = min(abs(v), 448.0)
    best, best_err = 0, None
    for c in range(0x7F):          # finite non-negative codes, 0x00 .. 0x7e
        err = abs(e4m3_value(c) - a)
        if best_err is None or err < best_err or (err == best_err and (c & 1) == 0 and (best & 1) == 1):
            best, best_err = c, err
    return sign | best


def e4m3_table() -> np.ndarray:
    """Values of all 256 E4M3 codes by e4m3_value (NaN at 0x7F and 0xFF)."""
    return np.array([e4m3_value(c) for c in range(256)])


def e4m3_encode_array(v) -> np.ndarray:
    """e4m3_encode of every element of v (uint8 codes of the same shape): the nearest of the finite
    non-negative values by a sorted search (they increase with the code), ties to the even code,
    magnitudes above 448 saturating, the sign bit taken from v (so -0.0 gives 0x80)."""
    v = np.asarray(v, np.float64)
    if np.isnan(v).any():
        raise ValueError("NaN has no E4M3 encoding here")
    vals = e4m3_table()[:0x7F]
    a = np.minimum(np.abs(v), 448.0)
    hi = np.minimum(np.searchsorted(vals, a, side="left"), 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    code = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def quantize_rows_e4m3(W, division: str = "f64") -> Dict[str, np.ndarray]:
    """Per-row scaled E4M3 codes of a weight matrix W [rows, cols]: scale_r = max_c |W_rc| / 448
    (1 for an all-zero row), codes_rc = e4m3(W_rc / scale_r); dequantised = value(code) * scale.

    division = "f64": the quotient W_rc / scale_r is taken in float64 and rounded once, to the
    code.  division = "f32": scale and quotient are IEEE float32 divisions (for W exactly
    representable in float32, such as bf16 weights), so a float32 implementation takes the same
    rounding decisions; the scale is the same either way (max|w| / 448 rounded once to float32).
    """
    W = np.asarray(W, np.float64)
    amax = np.abs(W).max(axis=1) if W.shape[1] else np.zeros(W.shape[0])
    if division == "f32":
        scale32 = np.where(amax > 0, amax.astype(np.float32) / np.float32(448.0), np.float32(1.0))
        scale32 = scale32.astype(np.float32)
        q = (W.astype(np.float32) / scale32[:, None]).astype(np.float64)
        scale = scale32.astype(np.float64)
    elif division == "f64":
        scale = np.where(amax > 0, amax / 448.0, 1.0).astype(np.float32).astype(np.float64)
        q = W / scale[:, None]
    else:
        raise ValueError(division)
    codes = e4m3_encode_array(q)
    return dict(codes=codes, scale=scale.astype(np.float32), dequantized=dequantize_rows_e4m3(codes, scale))


def dequantize_rows_e4m3(codes, scale) -> np.ndarray:
    """value(codes[..., r, c]) * scale[..., r] in float64 (exact: a 4-bit significand times a
    float32 scale)."""
    codes = np.asarray(codes)
    return e4m3_table()[codes.astype(np.int64)] * np.asarray(scale, np.float64)[..., None]


# ----------------------------------------------------------------------------- INT8 expert weights
# The mini-moe tutorial's deployment advice (model compression: quantise every expert to INT8 to
# cut what must be stored and loaded).  The pages give no scheme; the reading used is symmetric
# per-output-row scaling: scale_r = max_c |W_rc| / 127 (1 for an all-zero row) and
# q_rc = the integer nearest to W_rc / scale_r (ties to even), in [-127, 127].

def quantize_rows_int8(W) -> Dict[str, np.ndarray]:
    """Per-row symmetric INT8 codes of W [rows, cols].  The scale and the quotient are IEEE
    float32 divisions of the float32 values of W (exact for bf16 or fp32 weights), so a float32
    implementation takes the same rounding decisions; the quotient is rounded to the nearest
    integer, ties to even.  Returns codes (int8), scale (float32 [rows]) and the dequantised
    matrix codes * scale in float64."""
    W32 = np.asarray(W, np.float64).astype(np.float32)
    rows = W32.shape[0]
    amax = np.abs(W32).max(axis=1) if W32.shape[1] else np.zeros(rows, np.float32)
    scale = np.where(amax > 0, amax / np.float32(127.0), np.float32(1.0)).astype(np.float32)
    q = (W32 / scale[:, None]).astype(np.float32)
    codes = np.clip(np.rint(q), -127, 127).astype(np.int8)
    return dict(codes=codes, scale=scale, dequantized=dequantize_rows_int8(codes, scale))


def dequantize_rows_int8(codes, scale) -> np.ndarray:
    """codes[..., r, c] * scale[..., r] in float64 (exact)."""
    return np.asarray(codes, np.float64) * np.asarray(scale, np.float64)[..., None]


def quantize_experts(W, fmt: str, joint_blocks: bool = False) -> Dict[str, np.ndarray]:
    """Quantise a stack of expert matrices W [B, rows, cols] (fmt "int8" or "e4m3", float32
    division).  joint_blocks=False: every row of every block gets its own scale (scale [B, rows]).
    joint_blocks=True: row r of all B blocks together is one row of the [rows, B cols] matrix the
    blocks form side by side (the shared experts' down projections, which act as one wide expert),
    with one scale per r (scale [rows]).  Returns codes [B, rows, cols], scale and dequantized
    [B, rows, cols]."""
    W = np.asarray(W, np.float64)
    B, R, C = W.shape
    flat = np.concatenate(list(W), axis=1) if joint_blocks else W.reshape(B * R, C)
    q = quantize_rows_int8(flat) if fmt == "int8" else quantize_rows_e4m3(flat, "f32")
    if fmt not in ("int8", "e4m3"):
        raise ValueError(fmt)
    if joint_blocks:
        codes = np.stack([q["codes"][:, b * C:(b + 1) * C] for b in range(B)])
        deq = np.stack([q["dequantized"][:, b * C:(b + 1) * C] for b in range(B)])
        return dict(codes=codes, scale=q["scale"], dequantized=deq)
    return dict(codes=q["codes"].reshape(B, R, C), scale=q["scale"].reshape(B, R),
                dequantized=q["dequantized"].reshape(B, R, C))


# ----------------------------------------------------------------------------- whole layer
def moe_layer(inp: Dict, *, E: int, k: int, act: str, n_shared: int = 0, cf: float = 0.0,
              lb_coef: float = 0.01, z_coef: float = 0.001,
              tokens: Optional[Sequence[int]] = None, temperature: float = 1.0) -> Dict:
    """Forward pass of the layer on ``inp`` (the tensors of ``synth.make_inputs``).

    Routing, dispatch and losses are computed for every token; the FFNs and the combine only for
    ``tokens`` (all tokens when None).  With a router temperature the logits are divided by it
    before everything that follows (``temper``).  Returns routing, layout, losses and
    y [len(tokens), d]."""
    x = _f64(inp["x"])
    T = x.shape[0]
    z = router_logits(x, inp["w_router"], inp.get("logit_bias"))
    if temperature != 1.0:
        z = temper(z, temperature)
    P, lse = softmax_lse(z)
    idx = topk_select(z, k)
    w = renormalise(P, idx) if T else np.zeros((0, k))
    cap = capacity(cf, T, k, E)
    lay = dispatch(idx, E, cap)
    lb, zl = aux_losses(P, lse, lay["counts"], k, lb_coef, z_coef)
    if tokens is None:
        tokens = list(range(T))
    tokens = [int(t) for t in tokens]
    want = set(tokens)

    A = int(lay["offsets"][E])
    d = x.shape[1]
    y_perm = np.zeros((A, d))
    for e in range(E):
        lo, hi = int(lay["offsets"][e]), int(lay["offsets"][e + 1])
        rows = [r for r in range(lo, hi) if int(lay["tok_of"][r]) in want]
        if not rows:
            continue
        xr = x[lay["tok_of"][rows]]
        g = lambda name: None if inp.get(name) is None else inp[name][e]
        y_perm[rows] = expert_ffn(xr, act, g("w_up"), g("w_down"), g("w_gate"), g("b_up"), g("b_down"))

    y_shared = None
    if n_shared > 0:
        xs = x[tokens]
        y_shared = np.zeros((len(tokens), d))
        for s in range(n_shared):
            gs = None if inp.get("ws_gate") is None else inp["ws_gate"][s]
            y_shared += expert_ffn(xs, act, inp["ws_up"][s], inp["ws_down"][s], gs)
    y = combine(idx, w, lay["row_of"], y_perm, tokens, y_shared)
    return dict(z=z, P=P, lse=lse, idx=idx, w=w, gap=topk_gap(z, k), cap=cap, lb=lb, zl=zl,
                y=y, tokens=np.asarray(tokens, dtype=np.int64), y_perm=y_perm, **lay)
