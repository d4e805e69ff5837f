"""GPU backward of the expert FFNs (moe_expert_ffn_backward) against the oracle (needs a B300).

Expert level: the permuted rows, their offsets and row_of come from the oracle's own forward
routing, built into the library's layout on the CPU (rows past offsets[E] hold NaN, which must not
be read); the rows' upstream gradients dy_perm and the shared experts' dy are seeded draws in the
layer dtype, so the GPU and the oracle see bit-identical inputs.  fp32 layers differ only by fp32
arithmetic: every gradient within max|d| <= 1e-4 max|ref|.  bf16 layers contract on the tensor
cores with du, dg (or da) and h rounded to bf16 as operands: max|d| <= 1e-2 max|ref|.  dx starts
from a seeded fp32 array, to which the call must add.

Layer level: the forward steps, moe_combine_backward, moe_route_backward and this call in turn,
against the oracle's moe_layer_backward on the same inputs (the routing must agree: checked
first).  fp32 layers 1e-4 max|ref|; bf16 layers 2e-2 max|ref| (the forward's hidden rows and the
rows' upstream gradients are rounded to bf16 there, the oracle keeps them exact).
"""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_89_b300 import moe
from oracle import moe_backward as B
from oracle import moe_oracle as O
from synth import Workload, make_inputs

from parity_utils import run_steps, to_np

pytestmark = pytest.mark.gpu

CASES = {
    "bf16_swiglu_cap_shared": Workload("ebw_bf16_swiglu_cap", T=300, d=256, E=8, k=2, dff=128, act="swiglu",
                                       dtype="bf16", cf=1.0, n_shared=1, seed=71, wseed=71),
    "fp32_gelu_bias": Workload("ebw_fp32_gelu_bias", T=130, d=96, E=6, k=3, dff=64, act="gelu", dtype="f32",
                               bias=True, bias_std=0.3, seed=72, wseed=72),
    "bf16_gelu_bias_shared2": Workload("ebw_bf16_gelu_bias_sh2", T=160, d=128, E=16, k=4, dff=256, act="gelu",
                                       dtype="bf16", bias=True, bias_std=0.3, cf=1.25, n_shared=2, seed=73,
                                       wseed=73),
    "bf16_long_groups": Workload("ebw_bf16_long", T=600, d=256, E=4, k=2, dff=384, act="gelu", dtype="bf16",
                                 seed=74, wseed=74),
    "bf16_sparse_E64": Workload("ebw_bf16_sparse", T=8, d=128, E=64, k=2, dff=64, act="swiglu", dtype="bf16",
                                n_shared=1, seed=75, wseed=75),
    "fp32_swiglu_E64": Workload("ebw_fp32_swiglu_E64", T=200, d=192, E=64, k=6, dff=128, act="swiglu",
                                dtype="f32", n_shared=1, seed=76, wseed=76),
    # the largest expert count (256 groups in the tensor-core GEMM's tile table), top-8
    "bf16_E256_k8": Workload("ebw_bf16_E256_k8", T=96, d=128, E=256, k=8, dff=64, act="swiglu", dtype="bf16",
                             seed=77, wseed=77),
    # decode-shaped: 32 tokens, d = 2048 (32 K steps per tile), 64 experts, two shared experts
    "bf16_decode": Workload("ebw_bf16_decode", T=32, d=2048, E=64, k=6, dff=256, act="swiglu", dtype="bf16",
                            n_shared=2, seed=78, wseed=78),
}

# bf16 layers contract on the tensor cores with the operands the backward creates (du, dg or da,
# h) rounded to bf16 (relative 2^-9 each); fp32 layers stay fp32 throughout.
EXPERT_TOL = {"f32": 1e-4, "bf16": 1e-2}

GRAD_KEYS = ("dw_up", "dw_gate", "dw_down", "db_up", "db_down", "dws_up", "dws_gate", "dws_down")


def _close(got, ref, what, tol):
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    scale = max(float(np.abs(ref).max()), 1e-30)
    err = float(np.abs(got - ref).max()) / scale
    print(f"  {what}: max|d|/max|ref| {err:.2e}")
    assert err <= tol, (what, err)


def _grad_tensors(wl, dev):
    E, d, f, S = wl.E, wl.d, wl.dff, wl.n_shared
    z = dict(dtype=torch.float32, device=dev)
    g = {"dw_up": torch.full((E, f, d), float("nan"), **z), "dw_down": torch.full((E, d, f), float("nan"), **z)}
    if wl.act == "swiglu":
        g["dw_gate"] = torch.full((E, f, d), float("nan"), **z)
    if wl.bias:
        g["db_up"] = torch.full((E, f), float("nan"), **z)
        g["db_down"] = torch.full((E, d), float("nan"), **z)
    if S:
        g["dws_up"] = torch.full((S, f, d), float("nan"), **z)
        g["dws_down"] = torch.full((S, d, f), float("nan"), **z)
        if wl.act == "swiglu":
            g["dws_gate"] = torch.full((S, f, d), float("nan"), **z)
    return g


def _oracle_fwd(wl, inp_cpu):
    return O.moe_layer(inp_cpu, E=wl.E, k=wl.k, act=wl.act, n_shared=wl.n_shared, cf=wl.cf, lb_coef=wl.lb_coef,
                       z_coef=wl.z_coef, temperature=wl.temperature)


def _oracle_expert_grads(wl, inp_cpu, x_perm, offsets, row_of, dy_perm, dy, dx0):
    """The oracle's expert backward over given rows: per routed expert, then the scatter of the
    rows' input gradients, then the shared experts."""
    f64 = O._f64
    E, S = wl.E, wl.n_shared
    glu = wl.act == "swiglu"
    ref = {"dw_up": np.zeros(np.shape(inp_cpu["w_up"])), "dw_down": np.zeros(np.shape(inp_cpu["w_down"]))}
    if glu:
        ref["dw_gate"] = np.zeros(np.shape(inp_cpu["w_gate"]))
    if wl.bias:
        ref["db_up"] = np.zeros(np.shape(inp_cpu["b_up"]))
        ref["db_down"] = np.zeros(np.shape(inp_cpu["b_down"]))
    dx_rows = np.zeros_like(x_perm)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi <= lo:
            continue
        ge = B.expert_ffn_backward(x_perm[lo:hi], wl.act, dy_perm[lo:hi], f64(inp_cpu["w_up"][e]),
                                   f64(inp_cpu["w_down"][e]), f64(inp_cpu["w_gate"][e]) if glu else None,
                                   f64(inp_cpu["b_up"][e]) if wl.bias else None)
        for name in ref:
            ref[name][e] = ge[name]
        dx_rows[lo:hi] = ge["dx"]
    dx = dx0.copy()
    T, k = row_of.shape
    for t in range(T):
        for j in range(k):
            if row_of[t, j] >= 0:
                dx[t] += dx_rows[row_of[t, j]]
    if S:
        x = f64(inp_cpu["x"])
        ref["dws_up"] = np.zeros(np.shape(inp_cpu["ws_up"]))
        ref["dws_down"] = np.zeros(np.shape(inp_cpu["ws_down"]))
        if glu:
            ref["dws_gate"] = np.zeros(np.shape(inp_cpu["ws_gate"]))
        for s in range(S):
            gs = B.expert_ffn_backward(x, wl.act, dy, f64(inp_cpu["ws_up"][s]), f64(inp_cpu["ws_down"][s]),
                                       f64(inp_cpu["ws_gate"][s]) if glu else None)
            ref["dws_up"][s] = gs["dw_up"]
            ref["dws_down"][s] = gs["dw_down"]
            if glu:
                ref["dws_gate"][s] = gs["dw_gate"]
            dx = dx + gs["dx"]
    ref["dx"] = dx
    return ref


def _run_expert_backward(cfg, inp, x_perm, offsets, row_of, dy, dy_perm, grads, dx):
    scratch = torch.empty(max(moe.moe_expert_backward_scratch_size(cfg), 256), dtype=torch.uint8, device="cuda")
    moe.moe_expert_ffn_backward(cfg, moe.make_weights(inp), inp["x"], x_perm, offsets, row_of, dy, dy_perm,
                                moe.make_expert_grads(grads), dx, scratch)
    return scratch


@pytest.mark.parametrize("case", list(CASES))
def test_expert_backward_matches_oracle(case):
    wl = CASES[case]
    inp_cpu = make_inputs(wl, "cpu")
    inp = {k: (v.cuda() if v is not None else None) for k, v in inp_cpu.items()}
    cfg = moe.config_from_workload(wl)
    T, d, E = wl.T, wl.d, wl.E
    _, amax = moe.moe_capacity(cfg)
    fwd = _oracle_fwd(wl, inp_cpu)
    offsets = np.asarray(fwd["offsets"], np.int64)
    n_rows = int(offsets[E])
    tok_of = np.asarray(fwd["tok_of"], np.int64)[:n_rows]
    row_of = np.asarray(fwd["row_of"], np.int64)
    dt = inp_cpu["x"].dtype
    rows = max(amax, 1)
    x_perm_t = torch.full((rows, d), float("nan"), dtype=dt)
    x_perm_t[:n_rows] = inp_cpu["x"][torch.from_numpy(tok_of)]
    gen = torch.Generator().manual_seed(900 + wl.seed)
    dy_perm_t = torch.full((rows, d), float("nan"), dtype=dt)
    dy_perm_t[:n_rows] = torch.randn((n_rows, d), generator=gen).to(dt)
    dy_t = torch.randn((T, d), generator=gen).to(dt)
    dx0_t = torch.randn((T, d), generator=gen, dtype=torch.float32)

    grads = _grad_tensors(wl, "cuda")
    dx = dx0_t.cuda()
    i32 = dict(dtype=torch.int32, device="cuda")
    off_d = torch.tensor(offsets, **i32)
    row_of_d = torch.tensor(row_of, **i32)
    x_perm_d, dy_perm_d, dy_d = x_perm_t.cuda(), dy_perm_t.cuda(), dy_t.cuda()
    scratch = _run_expert_backward(cfg, inp, x_perm_d, off_d, row_of_d, dy_d, dy_perm_d, grads, dx)
    torch.cuda.synchronize()

    ref = _oracle_expert_grads(wl, inp_cpu, O._f64(x_perm_t[:max(n_rows, 0)]), offsets, row_of,
                               O._f64(dy_perm_t[:n_rows]), O._f64(dy_t), dx0_t.double().numpy())
    tol = EXPERT_TOL[wl.dtype]
    for name in GRAD_KEYS:
        if name in grads:
            _close(to_np(grads[name]), ref[name], name, tol)
    _close(to_np(dx), ref["dx"], "dx", tol)
    assert moe.moe_read_device_status(scratch) == moe.MOE_OK
    empty = [e for e in range(E) if offsets[e + 1] == offsets[e]]
    for e in empty:  # an expert with no rows: zero gradients, not left untouched
        assert torch.count_nonzero(grads["dw_up"][e]) == 0 and torch.count_nonzero(grads["dw_down"][e]) == 0

    # deterministic: a second call gives the same bits
    grads2 = _grad_tensors(wl, "cuda")
    dx2 = dx0_t.cuda()
    _run_expert_backward(cfg, inp, x_perm_d, off_d, row_of_d, dy_d, dy_perm_d, grads2, dx2)
    torch.cuda.synchronize()
    assert torch.equal(dx, dx2)
    for name in grads:
        assert torch.equal(grads[name], grads2[name]), name


LAYER_CASES = ("bf16_swiglu_cap_shared", "fp32_gelu_bias", "fp32_swiglu_E64")


@pytest.mark.parametrize("case", LAYER_CASES)
def test_layer_backward_chain_matches_oracle(case):
    wl = CASES[case]
    inp_cpu = make_inputs(wl, "cpu")
    inp = {k: (v.cuda() if v is not None else None) for k, v in inp_cpu.items()}
    st = run_steps(wl, inp)
    assert st["status"] == moe.MOE_OK
    fwd = _oracle_fwd(wl, inp_cpu)
    assert np.array_equal(st["row_of"].cpu().numpy(), np.asarray(fwd["row_of"])), "routing differs"
    cfg = moe.config_from_workload(wl)
    T, d, E, k = wl.T, wl.d, wl.E, wl.k
    gen = torch.Generator().manual_seed(800 + wl.seed)
    dy_t = torch.randn((T, d), generator=gen).to(inp_cpu["x"].dtype)
    dy = dy_t.cuda()
    dlb, dzl = 1.3, 0.7
    dw = torch.empty((T, k), dtype=torch.float32, device="cuda")
    dy_perm = torch.zeros_like(st["x_perm"])
    moe.moe_combine_backward(cfg, dy, st["y_perm"], st["row_of"], st["topk_w"], dw, dy_perm)
    dz = torch.empty((T, E), dtype=torch.float32, device="cuda")
    dwr = torch.empty((E, d), dtype=torch.float32, device="cuda")
    dx = torch.empty((T, d), dtype=torch.float32, device="cuda")
    moe.moe_route_backward(cfg, inp["x"], inp["w_router"], inp.get("logit_bias"), st["topk_idx"], st["topk_w"],
                           st["counts"], dw, dlb, dzl, dz, dwr, dx)
    grads = _grad_tensors(wl, "cuda")
    _run_expert_backward(cfg, inp, st["x_perm"], st["offsets"], st["row_of"], dy, dy_perm, grads, dx)
    torch.cuda.synchronize()

    inp64 = {name: O._f64(v) for name, v in inp_cpu.items()}  # exact widening of the drawn tensors
    ref = B.moe_layer_backward(inp64, O._f64(dy_t), E=E, k=k, act=wl.act, n_shared=wl.n_shared, cf=wl.cf,
                               lb_coef=wl.lb_coef, z_coef=wl.z_coef, dlb=dlb, dzl=dzl,
                               temperature=wl.temperature)
    tol = 1e-4 if wl.dtype == "f32" else 2e-2
    _close(to_np(dwr), ref["dw_router"], "dw_router", tol)
    _close(to_np(dx), ref["dx"], "dx", tol)
    for name in GRAD_KEYS:
        if name in grads:
            _close(to_np(grads[name]), ref[name], name, tol)


def test_expert_backward_empty_batch_and_arguments():
    wl = CASES["bf16_sparse_E64"].replace(T=0)
    inp = make_inputs(wl, "cuda")
    cfg = moe.config_from_workload(wl)
    grads = _grad_tensors(wl, "cuda")
    scratch = torch.empty(max(moe.moe_expert_backward_scratch_size(cfg), 256), dtype=torch.uint8, device="cuda")
    moe.moe_expert_ffn_backward(cfg, moe.make_weights(inp), None, None, None, None, None, None,
                                moe.make_expert_grads(grads), None, scratch)
    torch.cuda.synchronize()
    for name, t in grads.items():  # nothing to differentiate: every gradient is zero
        assert torch.count_nonzero(t) == 0, name
    L = moe.lib()
    full = moe.config_from_workload(CASES["bf16_sparse_E64"])
    # NULL weights / gradients, a backup expert and 8-bit weights are refused before any launch
    assert L.moe_expert_ffn_backward(ctypes.byref(full), None, None, None, None, None, None, None, None, None, None,
                                     None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_expert_ffn_backward(ctypes.byref(full), ctypes.byref(moe.make_weights(inp)), None, None, None,
                                     None, None, None, ctypes.byref(moe.make_expert_grads(grads)), None, None,
                                     None) == moe.MOE_ERR_INVALID_ARG
    n = ctypes.c_size_t(0)
    for bad in (CASES["bf16_sparse_E64"].replace(backup=True), CASES["bf16_sparse_E64"].replace(weights8="int8")):
        c = moe.config_from_workload(bad)
        assert L.moe_expert_backward_scratch_size(ctypes.byref(c), ctypes.byref(n)) == moe.MOE_ERR_UNSUPPORTED


def test_backward_from_the_fused_forward_workspace():
    """moe_layer_forward keeps its routing, rows and y_perm in the workspace; the backward calls fed
    from moe_workspace_views give the same bits as when fed from the forward steps."""
    wl = CASES["bf16_swiglu_cap_shared"]
    inp_cpu = make_inputs(wl, "cpu")
    inp = {k: (v.cuda() if v is not None else None) for k, v in inp_cpu.items()}
    cfg = moe.config_from_workload(wl)
    T, d, E, k = wl.T, wl.d, wl.E, wl.k
    dy = torch.randn((T, d), generator=torch.Generator().manual_seed(5)).to(inp_cpu["x"].dtype).cuda()

    def backward(topk_idx, topk_w, counts, offsets, row_of, x_perm, y_perm):
        dw = torch.empty((T, k), dtype=torch.float32, device="cuda")
        dy_perm = torch.zeros(x_perm_shape, dtype=inp["x"].dtype, device="cuda")
        moe.moe_combine_backward(cfg, dy, y_perm, row_of, topk_w, dw, dy_perm)
        dz = torch.empty((T, E), dtype=torch.float32, device="cuda")
        dwr = torch.empty((E, d), dtype=torch.float32, device="cuda")
        dx = torch.empty((T, d), dtype=torch.float32, device="cuda")
        moe.moe_route_backward(cfg, inp["x"], inp["w_router"], inp.get("logit_bias"), topk_idx, topk_w, counts, dw,
                               1.0, 1.0, dz, dwr, dx)
        grads = _grad_tensors(wl, "cuda")
        _run_expert_backward(cfg, inp, x_perm, offsets, row_of, dy, dy_perm, grads, dx)
        torch.cuda.synchronize()
        return dict(dw=dw, dz=dz, dw_router=dwr, dx=dx, **grads)

    st = run_steps(wl, inp)
    x_perm_shape = tuple(st["x_perm"].shape)
    ref = backward(st["topk_idx"], st["topk_w"], st["counts"], st["offsets"], st["row_of"], st["x_perm"],
                   st["y_perm"])
    layer = moe.MoELayer(cfg, inp)
    _, _, counts, _ = layer.forward(inp["x"])
    v = moe.moe_workspace_views(cfg, layer.ws)
    got = backward(v["topk_idx"], v["topk_w"], counts, v["offsets"], v["row_of"], v["x_perm"], v["y_perm"])
    for name in ref:
        assert torch.equal(ref[name], got[name]), name
