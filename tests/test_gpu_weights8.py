"""8-bit expert weights on the GPU against the oracle (needs a B300).

The mini-moe tutorial (deployment optimisation) suggests quantising every expert to INT8; E4M3 is
the second 8-bit format.  Two checks:
  * moe_quantize_experts writes the codes and row scales of oracle.quantize_experts bit for bit
    (both take their decisions on IEEE float32 quotients);
  * the layer with 8-bit experts equals the oracle's layer run on the dequantised weights
    (codes x scale, exact in float64), within the bf16 output tolerance of every other layer.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_89_b300 import moe
from oracle import moe_oracle as O
from synth import WORKLOADS, Workload, make_inputs

from parity_utils import check_losses, check_output, oracle, run_layer, run_steps, to_np

pytestmark = pytest.mark.gpu

FORMATS = ["int8", "e4m3"]
# weight key -> (scale key, one scale per row over the blocks side by side)
QUANT = {"w_up": ("s_up", False), "w_gate": ("s_gate", False), "w_down": ("s_down", False),
         "ws_up": ("ss_up", False), "ws_gate": ("ss_gate", False), "ws_down": ("ss_down", True),
         "wb_up": ("sb_up", False), "wb_gate": ("sb_gate", False), "wb_down": ("sb_down", False)}


def _codes_np(t):
    return t.cpu().numpy()


def quantize_both(inp_cpu, inp_gpu, fmt):
    """Quantise on the GPU (the library) and on the CPU (the oracle); check that codes and scales
    agree bit for bit; return the GPU layer inputs and the oracle's inputs with dequantised
    weights."""
    q_gpu = moe.quantize_expert_tensors(inp_gpu, fmt)
    deq = dict(inp_cpu)
    for wk, (sk, joint) in QUANT.items():
        w = inp_cpu.get(wk)
        if w is None:
            continue
        w3 = w.reshape(1, *w.shape) if w.dim() == 2 else w
        ref = O.quantize_experts(O._f64(w3), fmt, joint_blocks=joint)
        got_codes = _codes_np(q_gpu[wk]).reshape(w3.shape)
        ref_codes = ref["codes"].astype(np.int8) if fmt == "int8" else ref["codes"]
        assert np.array_equal(got_codes.view(np.uint8), ref_codes.view(np.uint8)), (wk, fmt)
        got_scale = q_gpu[sk].cpu().numpy().reshape(ref["scale"].shape)
        assert np.array_equal(got_scale, ref["scale"]), (sk, fmt)
        deq[wk] = ref["dequantized"].reshape(w.shape)
    return q_gpu, deq


def test_quantize_matches_oracle_special_values():
    """Zero rows, exact halves of the INT8 step, saturating and tiny E4M3 quotients, and -0.0; a
    non-finite weight is counted."""
    rng = np.random.default_rng(40)
    W = rng.standard_normal((3, 70, 96)) * 0.02
    W[0, 5] = 0.0
    s = 2.0 ** -7
    W[1, 9, :8] = np.array([127, 0.5, 1.5, 2.5, -2.5, -0.5, 126.5, -0.0]) * s   # int8 ties
    W[2, 3, :6] = [1e-9, -1e-9, 3.0, -3.0, 2.0 ** -20, -0.0]                    # e4m3 range ends
    Wb = torch.tensor(W, dtype=torch.float32).to(torch.bfloat16)
    for fmt in FORMATS:
        for joint in (False, True):
            B, R, C = Wb.shape
            blocks, rows = (B, R) if joint else (1, B * R)
            codes = torch.empty((B, R, C), dtype=torch.uint8, device="cuda")
            scale = torch.empty(rows, dtype=torch.float32, device="cuda")
            bad = torch.zeros(1, dtype=torch.int32, device="cuda")
            moe.moe_quantize_experts(Wb.cuda(), fmt, blocks, rows, C, codes, scale, bad)
            ref = O.quantize_experts(Wb.double().numpy(), fmt, joint_blocks=joint)
            assert np.array_equal(codes.cpu().numpy(), ref["codes"].view(np.uint8)), (fmt, joint)
            assert np.array_equal(scale.cpu().numpy(), ref["scale"].reshape(-1)), (fmt, joint)
            assert int(bad.item()) == 0
    # fp32 weights, and a non-finite weight counted (its row's codes are then meaningless)
    W32 = torch.tensor(W[:1], dtype=torch.float32)
    W32[0, 2, 7] = float("nan")
    W32[0, 4, 1] = float("inf")
    codes = torch.empty(W32.shape, dtype=torch.uint8, device="cuda")
    scale = torch.empty(70, dtype=torch.float32, device="cuda")
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_quantize_experts(W32.cuda(), "int8", 1, 70, 96, codes, scale, bad)
    assert int(bad.item()) == 2
    clean = [r for r in range(70) if r not in (2, 4)]
    ref = O.quantize_rows_int8(W32[0].double().numpy()[clean])
    assert np.array_equal(codes.cpu().numpy()[0][clean], ref["codes"].view(np.uint8))
    assert np.array_equal(scale.cpu().numpy()[clean], ref["scale"])


def test_quantize_rejects_bad_arguments():
    w = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    codes = torch.empty((4, 64), dtype=torch.uint8, device="cuda")
    scale = torch.empty(4, dtype=torch.float32, device="cuda")
    L = moe.lib()
    assert L.moe_quantize_experts(w.data_ptr(), moe.MOE_BF16, 0, 1, 4, 64, codes.data_ptr(), scale.data_ptr(),
                                  None, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_quantize_experts(w.data_ptr(), moe.MOE_BF16, 1, 1, -4, 64, codes.data_ptr(), scale.data_ptr(),
                                  None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_quantize_experts(None, moe.MOE_BF16, 1, 1, 4, 64, codes.data_ptr(), scale.data_ptr(),
                                  None, None) == moe.MOE_ERR_INVALID_ARG


LAYER_CASES = {
    # many rows per expert (256-token tiles), shared experts, capacity drops
    "swiglu_shared_cap": Workload("w8_swiglu_shared_cap", T=700, d=512, E=16, k=4, dff=256, act="swiglu",
                                  dtype="bf16", n_shared=2, cf=1.25, seed=41, wseed=41),
    # decode-sized call (32-token tiles), three shared experts whose down rows share one scale
    "swiglu_decode_shared3": Workload("w8_swiglu_decode_shared3", T=32, d=512, E=16, k=4, dff=256, act="swiglu",
                                      dtype="bf16", n_shared=3, seed=42, wseed=42),
    # GELU experts with biases (the 16-warp epilogue beside the converter warps), ragged tails
    "gelu_bias_ragged": Workload("w8_gelu_bias_ragged", T=1000, d=256, E=8, k=2, dff=512, act="gelu",
                                 dtype="bf16", bias=True, bias_std=0.02, cf=1.1, seed=43, wseed=43),
    # a backup expert for the assignments over capacity, decode-sized
    "decode_backup": Workload("w8_decode_backup", T=32, d=256, E=8, k=2, dff=256, act="swiglu", dtype="bf16",
                              n_shared=1, cf=0.5, seed=44, wseed=44, backup=True),
}


def _backup_of(inp):
    return {n: inp.get(m) for n, m in (("w_up", "wb_up"), ("w_gate", "wb_gate"), ("w_down", "wb_down"),
                                       ("b_up", "bb_up"), ("b_down", "bb_down"))}


def check_layer8(wl, fmt, tokens=None):
    inp_cpu = make_inputs(wl, "cpu")
    inp_gpu = {k: (v.cuda() if v is not None else None) for k, v in inp_cpu.items()}
    q_gpu, deq = quantize_both(inp_cpu, inp_gpu, fmt)
    wl8 = wl.replace(weights8=fmt)
    if wl.backup:
        ref = O.moe_layer_backup_expert(deq, _backup_of(deq), E=wl.E, k=wl.k, act=wl.act, n_shared=wl.n_shared,
                                        cf=wl.cf, lb_coef=wl.lb_coef, z_coef=wl.z_coef)
    else:
        ref = oracle(wl, deq, tokens=tokens)
    assert (ref["gap"] >= 1e-5).all()
    lay = run_layer(wl8, q_gpu)
    assert lay["status"] == moe.MOE_OK, moe.moe_status_string(lay["status"])
    toks = ref["tokens"] if "tokens" in ref else np.arange(wl.T)
    check_output(to_np(lay["y"])[toks], ref["y"], "bf16", f"y ({fmt})")
    check_losses(lay["losses"], ref["lb"], ref["zl"])
    steps = run_steps(wl8, q_gpu)
    assert steps["status"] == moe.MOE_OK
    assert torch.equal(steps["y"], lay["y"])
    return lay, ref


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("case", list(LAYER_CASES))
def test_layer_weights8_matches_oracle(case, fmt):
    check_layer8(LAYER_CASES[case], fmt)


@pytest.mark.parametrize("fmt", FORMATS)
def test_full_decode_weights8(fmt):
    """The decode-shaped call (32 tokens, 64 routed + 2 shared SwiGLU experts, d 2048) with 8-bit
    experts, all tokens, in the launch configuration the benchmark times."""
    check_layer8(WORKLOADS["decode_bf16"], fmt)


def test_weights8_argument_checks():
    wl = LAYER_CASES["swiglu_decode_shared3"].replace(weights8="int8")
    inp = make_inputs(wl, "cuda")
    q = moe.quantize_expert_tensors(inp, "int8")
    cfg = moe.config_from_workload(wl)
    ws = moe.alloc_workspace(cfg)
    y = torch.empty_like(inp["x"])
    losses = torch.empty(2, dtype=torch.float32, device="cuda")
    L = moe.lib()
    import ctypes
    no_scale = dict(q, ss_down=None)
    w = moe.make_weights(no_scale)
    st = L.moe_layer_forward(ctypes.byref(cfg), ctypes.byref(w), inp["x"].data_ptr(), y.data_ptr(),
                             losses.data_ptr(), None, None, ws.data_ptr(), None)
    assert st == moe.MOE_ERR_INVALID_ARG
    cfg32 = moe.config_from_workload(wl.replace(dtype="f32"))
    assert L.moe_workspace_size(ctypes.byref(cfg32), ctypes.byref(ctypes.c_size_t())) == moe.MOE_ERR_UNSUPPORTED
    bad = moe.config_from_workload(wl)
    bad.expert_weights = 3
    assert L.moe_workspace_size(ctypes.byref(bad), ctypes.byref(ctypes.c_size_t())) == moe.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("fmt", FORMATS)
def test_weights8_deterministic_and_graph_replay(fmt):
    """Repeat calls give the same bits, and a CUDA-graph replay of the layer equals the eager call
    (the converter warps and the stage barriers do not depend on scheduling)."""
    wl = LAYER_CASES["swiglu_decode_shared3"].replace(weights8=fmt)
    inp = make_inputs(wl, "cuda")
    q = moe.quantize_expert_tensors(inp, fmt)
    layer = moe.MoELayer(moe.config_from_workload(wl), q)
    y0, l0, c0, d0 = layer.forward(inp["x"])
    y1, l1, c1, d1 = layer.forward(inp["x"])
    assert torch.equal(y0, y1) and torch.equal(l0, l1) and torch.equal(c0, c1)
    cfg = layer.cfg
    y = torch.empty_like(inp["x"])
    losses = torch.empty(2, dtype=torch.float32, device="cuda")
    counts = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
    drops = torch.empty(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        moe.moe_layer_forward(cfg, layer.weights, inp["x"], y, losses, counts, drops, layer.ws, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.moe_layer_forward(cfg, layer.weights, inp["x"], y, losses, counts, drops, layer.ws,
                              torch.cuda.current_stream())
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, y0) and torch.equal(losses, l0)
    assert moe.moe_read_device_status(layer.ws) == moe.MOE_OK
