"""The C-ABI library builds, loads and exports every symbol ``include/moe.h`` declares; host-only
entry points (validation, capacity, workspace size, launch count) behave as documented.
No call here touches a GPU."""
import ctypes
import os
import re

import pytest

from mixture_experts_layer_89_b300 import build, moe
from oracle import moe_oracle as O
from synth import WORKLOADS

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return moe.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^[a-z_0-9 \*]*?\b(moe_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("moe_route", "moe_permute", "moe_expert_ffn", "moe_combine", "moe_layer_forward"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(moe.EXPORTED)


def test_status_strings(L):
    for s in (0, -1, -2, -3, -4, -5):
        assert moe.moe_status_string(s)
    assert moe.moe_status_string(0) == "ok"


@pytest.mark.parametrize("cf,T,k,E", [(1.25, 8192, 2, 16), (1.0, 16384, 2, 128), (1.0, 10, 1, 3), (0.5, 3, 1, 1),
                                      (0.1, 10, 1, 1), (0.3, 1000, 2, 7), (2.0, 5, 3, 4), (1e-30, 7, 1, 2),
                                      (1e30, 7, 2, 2), (0.0, 9, 2, 4), (-1.0, 9, 2, 4), (1.25, 1, 1, 8)])
def test_capacity_matches_oracle(L, cf, T, k, E):
    cfg = moe.make_config(T, 64, E, k, 128, dtype="f32", capacity_factor=cf)
    cap, amax = moe.moe_capacity(cfg)
    ref = O.capacity(cf, T, k, E)
    if ref is None:
        assert cap == -1 and amax == T * k
    else:
        # the library clamps capacities above T k (no assignment can drop either way)
        assert cap == min(ref, T * k)
        assert amax == min(T * k, E * min(ref, T * k))


def test_workspace_grows_with_shape(L):
    small = moe.moe_workspace_size(moe.make_config(64, 64, 8, 2, 128, dtype="f32"))
    big = moe.moe_workspace_size(moe.config_from_workload(WORKLOADS["finegrained_bf16"]))
    assert 0 < small < big
    assert big % 256 == 0


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), moe.MOE_ERR_INVALID_ARG),
    (dict(E=0), moe.MOE_ERR_INVALID_ARG),
    (dict(k=3, E=2), moe.MOE_ERR_UNSUPPORTED),
    (dict(k=9, E=16), moe.MOE_ERR_UNSUPPORTED),
    (dict(E=257), moe.MOE_ERR_UNSUPPORTED),
    (dict(d=96, dtype="bf16"), moe.MOE_ERR_UNSUPPORTED),
    (dict(dff=96, dtype="bf16"), moe.MOE_ERR_UNSUPPORTED),
    (dict(act="swiglu", has_bias=True), moe.MOE_ERR_UNSUPPORTED),
    (dict(n_shared=2, dff=192, act="swiglu", dtype="bf16"), moe.MOE_ERR_UNSUPPORTED),
])
def test_invalid_configs_rejected_on_host(L, kw, status):
    base = dict(T=64, d=64, E=8, k=2, dff=128, dtype="f32")
    base.update(kw)
    cfg = moe.make_config(**base)
    n = ctypes.c_size_t(0)
    assert L.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == status
    # every entry point validates before it touches the device
    assert L.moe_route(ctypes.byref(cfg), None, None, None, None, None, None, None, None, None) == status
    assert L.moe_layer_forward_launches(ctypes.byref(cfg)) == -1


def test_null_pointers_rejected_on_host(L):
    cfg = moe.make_config(64, 64, 8, 2, 128, dtype="f32")
    assert L.moe_route(ctypes.byref(cfg), None, None, None, None, None, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_layer_forward(ctypes.byref(cfg), None, None, None, None, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    w = moe.MoeWeights()
    assert L.moe_expert_ffn(ctypes.byref(cfg), None, None, ctypes.byref(w), None, None, None, None, None) == \
        moe.MOE_ERR_INVALID_ARG
    ev = (ctypes.c_void_p * 3)()
    assert L.moe_layer_forward_timed(ctypes.byref(cfg), None, None, None, None, None, None, None, None, ev, 3) == \
        moe.MOE_ERR_INVALID_ARG
    assert L.moe_read_device_status(None, None) == moe.MOE_ERR_INVALID_ARG


def test_misaligned_pointer_rejected_on_host(L):
    cfg = moe.make_config(64, 64, 8, 2, 128, dtype="f32")
    ptr = 0x10000008  # never dereferenced: alignment is checked first
    assert L.moe_route(ctypes.byref(cfg), ptr, 0x10000000, None, 0x20000000, 0x30000000, 0x40000000, 0x50000000,
                       0x60000000, None) == moe.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_launch_count(L, name):
    wl = WORKLOADS[name]
    n = moe.moe_layer_forward_launches(moe.config_from_workload(wl))
    # bf16: one tensor-core router launch whose last CTA also scans the dispatch histograms, then the
    # rank kernel and the row gather; fp32: router + reduction, histogram + scan + rank + gather
    router, dispatch = (1, 2) if wl.dtype == "bf16" else (2, 4)
    # bf16: the up and the down projection each carry the routed and the shared experts in one
    # launch; fp32: routed up + down, then shared up + down
    ffn = 2 if wl.dtype == "bf16" else 2 + (2 if wl.n_shared else 0)
    assert n == router + dispatch + ffn + 1
    assert moe.moe_layer_forward_launches(moe.config_from_workload(wl, T=0)) == (1 if wl.dtype == "bf16" else 2)


def test_wait_limit_setter_rejects_bad_workspace_on_host(L):
    assert L.moe_set_wait_limit(None, 5, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_set_wait_limit((1 << 12) + 8, 5, None) == moe.MOE_ERR_INVALID_ARG   # misaligned, never touched
