"""GPU backward of the routing half of the layer against the oracle (needs a B300).

moe_combine_backward and moe_route_backward (both of its paths: fp32 CUDA cores, and the tensor
cores with dz split into bf16 hi + lo parts) run on the forward steps' own outputs (routing,
rows, y_perm from moe_route / moe_permute / moe_expert_ffn); the oracle's combine_backward and
router_backward get the same routing and rows (so near-tie tokens need no exemption), and its own
fp64 logits for the softmax.  Acceptance: fp32 gradients normwise, max|d| <= 1e-4 max|ref|; the
rows' upstream gradients w_tj dy_t within the rounding of the fp32 product to the layer dtype.
"""
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
    "bf16_swiglu_cap": Workload("bw_bf16_swiglu_cap", T=300, d=256, E=8, k=2, dff=128, act="swiglu", dtype="bf16",
                                cf=1.0, n_shared=1, seed=61, wseed=61),
    "fp32_gelu_bias": Workload("bw_fp32_gelu_bias", T=130, d=96, E=6, k=3, dff=64, act="gelu", dtype="f32",
                               bias=True, seed=62, wseed=62),
    "bf16_temp2_E64": Workload("bw_bf16_temp2_E64", T=200, d=512, E=64, k=6, dff=128, act="swiglu", dtype="bf16",
                               seed=63, wseed=63, temperature=2.0, logit_bias0=1.0),
    "bf16_decode": Workload("bw_bf16_decode", T=32, d=2048, E=64, k=6, dff=128, act="swiglu", dtype="bf16",
                            n_shared=2, seed=64, wseed=64),
    "bf16_E256_k8": Workload("bw_bf16_E256_k8", T=96, d=128, E=256, k=8, dff=64, act="swiglu", dtype="bf16",
                             seed=65, wseed=65),
}


def _close(got, ref, what, tol=1e-4):
    scale = max(float(np.abs(ref).max()), 1e-30)
    err = float(np.abs(got - ref).max()) / scale
    print(f"  {what}: max|d|/max|ref| {err:.2e}")
    assert err <= tol, (what, err)


@pytest.mark.parametrize("case", list(CASES))
def test_routing_backward_matches_oracle(case):
    wl = CASES[case]
    inp_cpu = make_inputs(wl, "cpu")
    inp = {k: (v.cuda() if v is not None else None) for k, v in inp_cpu.items()}
    st = run_steps(wl, inp)
    assert st["status"] == moe.MOE_OK
    cfg = moe.config_from_workload(wl)
    T, d, E, k = wl.T, wl.d, wl.E, wl.k
    g = torch.Generator(device="cuda").manual_seed(700 + wl.seed)
    dy = torch.randn((T, d), generator=g, device="cuda").to(inp["x"].dtype)
    dw = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    dy_perm = torch.zeros_like(st["x_perm"])
    moe.moe_combine_backward(cfg, dy, st["y_perm"], st["row_of"], st["topk_w"], dw, dy_perm)
    dlb, dzl = 1.3, 0.7
    torch.cuda.synchronize()

    row_of = st["row_of"].cpu().numpy()
    tw = st["topk_w"].cpu().numpy().astype(np.float64)
    cb = B.combine_backward(to_np(dy), to_np(st["y_perm"]), row_of, tw)
    _close(to_np(dw), cb["dw"], "dw")
    kept = row_of[row_of >= 0]
    got_rows = to_np(dy_perm)[kept]
    ref_rows = cb["dy_perm"][kept]
    if wl.dtype == "bf16":
        _, ex = np.frexp(np.abs(ref_rows))
        # the product is rounded to fp32, then to bf16: half a bf16 ulp plus the fp32 rounding
        bound = np.ldexp(1.0, ex - 9) + np.abs(ref_rows) * 2.0 ** -23
        assert (np.abs(got_rows - ref_rows) <= bound).all(), float((np.abs(got_rows - ref_rows) / bound).max())
    else:
        _close(got_rows, ref_rows, "dy_perm", 1e-6)
    z = O.router_logits(O._f64(inp_cpu["x"]), inp_cpu["w_router"], inp_cpu.get("logit_bias"))
    P, lse = O.softmax_lse(O.temper(z, wl.temperature))
    rb = B.router_backward(O._f64(inp_cpu["x"]), O._f64(inp_cpu["w_router"]), P, lse,
                           st["topk_idx"].cpu().numpy(), tw, to_np(dw), st["counts"].cpu().numpy(), E=E, k=k,
                           lb_coef=wl.lb_coef, z_coef=wl.z_coef, dlb=dlb, dzl=dzl, temperature=wl.temperature)
    n_scratch = moe.moe_route_backward_scratch_size(cfg)
    # bf16 layers with E a multiple of 64 have a tensor-core path (taken when a scratch is given);
    # every layer has the CUDA-core one
    assert (n_scratch > 0) == (wl.dtype == "bf16" and E % 64 == 0)
    for scratch in ([None, torch.empty(n_scratch, dtype=torch.uint8, device="cuda")] if n_scratch else [None]):
        path = "CUDA cores" if scratch is None else "tensor cores"
        outs = []
        for _ in range(2):  # deterministic: a second call gives the same bits
            dz = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
            dwr = torch.full((E, d), float("nan"), dtype=torch.float32, device="cuda")
            dx = torch.full((T, d), float("nan"), dtype=torch.float32, device="cuda")
            moe.moe_route_backward(cfg, inp["x"], inp["w_router"], inp.get("logit_bias"), st["topk_idx"],
                                   st["topk_w"], st["counts"], dw, dlb, dzl, dz, dwr, dx, scratch)
            torch.cuda.synchronize()
            outs.append((dz, dwr, dx))
        dz, dwr, dx = outs[0]
        print(f"  {path}:")
        _close(to_np(dz), rb["dz"], "dz")
        _close(to_np(dwr), rb["dw_router"], "dw_router")
        _close(to_np(dx), rb["dx"], "dx")
        assert all(torch.equal(a, b) for a, b in zip(outs[0], outs[1]))
        if scratch is not None:
            assert moe.moe_read_device_status(scratch) == moe.MOE_OK


def test_routing_backward_empty_batch_and_arguments():
    wl = CASES["bf16_swiglu_cap"].replace(T=0)
    inp = make_inputs(wl, "cuda")
    cfg = moe.config_from_workload(wl)
    dwr = torch.full((wl.E, wl.d), float("nan"), dtype=torch.float32, device="cuda")
    counts = torch.zeros(wl.E, dtype=torch.int32, device="cuda")
    moe.moe_route_backward(cfg, None, inp["w_router"], None, None, None, counts, None, 1.0, 1.0, None, dwr, None)
    moe.moe_combine_backward(cfg, None, None, None, None, None, None)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dwr) == 0
    import ctypes
    L = moe.lib()
    assert L.moe_route_backward(ctypes.byref(moe.config_from_workload(CASES["bf16_swiglu_cap"])), None, None, None,
                                None, None, None, None, 1.0, 1.0, None, None, None, None,
                                None) == moe.MOE_ERR_INVALID_ARG
