"""Host-side logic of the backward entry points (no GPU needed: every call here returns before any
device work): the scratch sizes, the refusals, and the argument checks.

The scratch layouts are restated here from their definitions in moe.h (each buffer rounded up to
256 bytes), so a change of either side shows up as a mismatch.
"""
import ctypes

import pytest

from mixture_experts_layer_89_b300 import moe
from synth import WORKLOADS


def _r256(n):
    return (n + 255) // 256 * 256


def _r64(n):
    return (n + 63) // 64 * 64


def _expert_scratch(wl):
    cfg = moe.config_from_workload(wl)
    _, A = moe.moe_capacity(cfg)
    glu = wl.act == "swiglu"
    f, d, E, T, S = wl.dff, wl.d, wl.E, wl.T, wl.n_shared
    R = max(A, T if S else 0)
    Kd = 2 * f if glu else f
    tc = wl.dtype == "bf16"
    Kp = max(_r64(A + 63 * E) if A > 0 else 0, _r64(T) if S else 0) if tc else 0
    parts = [256, R * f * 4, R * f * 4 if glu else 0, R * f * 4, A * d * 4]
    if tc:
        parts += [(E + 1) * 4, R * Kd * 2, R * f * 2, Kd * Kp * 2, f * Kp * 2, d * Kp * 2, d * Kp * 2]
    return sum(_r256(p) for p in parts)


def _route_scratch(wl):
    if wl.dtype != "bf16" or wl.E % 64 or wl.T <= 0:
        return 0
    Tp, E, d, T = _r64(wl.T), wl.E, wl.d, wl.T
    slices = 8  # the token slices the dW_r contraction may be split into
    return sum(_r256(p) for p in (256, T * 2 * E * 2, 2 * E * Tp * 2, d * Tp * 2, slices * 2 * E * d * 4,
                                  (slices + 1) * 4))


NAMES = ["tiny_fp32", "flash_bf16", "finegrained_bf16", "decode_bf16", "skewed_bf16", "skewed_cf1_bf16"]


@pytest.mark.parametrize("name", NAMES)
def test_backward_scratch_sizes(name):
    wl = WORKLOADS[name]
    cfg = moe.config_from_workload(wl)
    assert moe.moe_expert_backward_scratch_size(cfg) == _expert_scratch(wl)
    assert moe.moe_route_backward_scratch_size(cfg) == _route_scratch(wl)


def test_route_scratch_only_where_the_tensor_cores_apply():
    base = WORKLOADS["finegrained_bf16"]
    assert moe.moe_route_backward_scratch_size(moe.config_from_workload(base)) > 0       # E = 64
    for wl in (base.replace(E=48), base.replace(dtype="f32"), base.replace(T=0)):
        assert moe.moe_route_backward_scratch_size(moe.config_from_workload(wl)) == 0


def test_expert_backward_refusals_and_argument_checks():
    L = moe.lib()
    n = ctypes.c_size_t(0)
    base = WORKLOADS["finegrained_bf16"].replace(T=64)
    for bad in (base.replace(backup=True), base.replace(weights8="int8"), base.replace(weights8="e4m3")):
        c = moe.config_from_workload(bad)
        assert L.moe_expert_backward_scratch_size(ctypes.byref(c), ctypes.byref(n)) == moe.MOE_ERR_UNSUPPORTED
        assert L.moe_expert_ffn_backward(ctypes.byref(c), None, None, None, None, None, None, None, None, None, None,
                                         None) == moe.MOE_ERR_UNSUPPORTED
    cfg = moe.config_from_workload(base)
    fake = 1 << 12  # 16-byte aligned, never dereferenced: every call below is refused first
    w = moe.MoeWeights()
    g = moe.MoeExpertGrads()
    # no weights / no gradients
    assert L.moe_expert_ffn_backward(ctypes.byref(cfg), None, fake, fake, fake, fake, fake, fake, ctypes.byref(g),
                                     fake, fake, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_expert_ffn_backward(ctypes.byref(cfg), ctypes.byref(w), fake, fake, fake, fake, fake, fake,
                                     ctypes.byref(g), fake, fake, None) == moe.MOE_ERR_INVALID_ARG
    # a misaligned input row pointer
    for k in ("w_up", "w_gate", "w_down", "ws_up", "ws_gate", "ws_down"):
        setattr(w, k, fake)
    for k in ("dw_up", "dw_gate", "dw_down", "dws_up", "dws_gate", "dws_down"):
        setattr(g, k, fake)
    assert L.moe_expert_ffn_backward(ctypes.byref(cfg), ctypes.byref(w), fake, fake + 2, fake, fake, fake, fake,
                                     ctypes.byref(g), fake, fake, None) == moe.MOE_ERR_INVALID_ARG
    # no scratch (it holds the status word)
    assert L.moe_expert_ffn_backward(ctypes.byref(cfg), ctypes.byref(w), fake, fake, fake, fake, fake, fake,
                                     ctypes.byref(g), fake, None, None) == moe.MOE_ERR_INVALID_ARG


def test_route_backward_argument_checks():
    L = moe.lib()
    cfg = moe.config_from_workload(WORKLOADS["finegrained_bf16"].replace(T=64))
    fake = 1 << 12
    args = [fake] * 7
    # non-finite loss weights, a misaligned scratch, missing outputs
    assert L.moe_route_backward(ctypes.byref(cfg), *args, float("nan"), 1.0, fake, fake, fake, None,
                                None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_route_backward(ctypes.byref(cfg), *args, 1.0, 1.0, fake, fake, fake, fake + 8,
                                None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_route_backward(ctypes.byref(cfg), *args, 1.0, 1.0, None, fake, fake, None,
                                None) == moe.MOE_ERR_INVALID_ARG


def test_workspace_views_lie_inside_the_workspace_and_do_not_overlap():
    for name in ("flash_bf16", "decode_bf16", "tiny_fp32"):
        wl = WORKLOADS[name]
        cfg = moe.config_from_workload(wl)
        base = 1 << 20  # 256-byte aligned, never dereferenced: the call is pointer arithmetic only
        size = moe.moe_workspace_size(cfg)
        v = moe.moe_workspace_views(cfg, base)
        _, A = moe.moe_capacity(cfg)
        elt = 2 if wl.dtype == "bf16" else 4
        extent = {"topk_idx": wl.T * wl.k * 4, "topk_w": wl.T * wl.k * 4, "counts": wl.E * 4,
                  "offsets": (wl.E + 1) * 4, "row_of": wl.T * wl.k * 4, "tok_of": A * 4, "x_perm": A * wl.d * elt,
                  "y_perm": A * wl.d * 4}
        spans = sorted((v[n], v[n] + extent[n], n) for n in extent)
        for lo, hi, n in spans:
            assert base <= lo and hi <= base + size and lo % 16 == 0, (name, n)
        for (lo0, hi0, n0), (lo1, hi1, n1) in zip(spans, spans[1:]):
            assert hi0 <= lo1, (name, n0, n1)
    L = moe.lib()
    cfg = moe.config_from_workload(WORKLOADS["flash_bf16"])
    out = moe.MoeForwardViews()
    assert L.moe_workspace_views(ctypes.byref(cfg), None, ctypes.byref(out)) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_workspace_views(ctypes.byref(cfg), (1 << 20) + 4, ctypes.byref(out)) == moe.MOE_ERR_INVALID_ARG
