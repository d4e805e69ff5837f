"""moe_route_noalloc: the router entry point that takes no workspace.

Some callers cannot allocate device memory at the time they route tokens: an engine that reserves
all of HBM for weights and caches at start-up and forbids later cudaMalloc calls, or a plug-in
running inside another framework's operator without access to that framework's allocator.  For
them the library keeps the router's scratch in a fixed device array of its own.  These tests check
that the variant gives the same results as moe_route with a caller-supplied workspace, over several
calls in a row (the array keeps each call's leftovers), and that over-large shapes are refused on
the host.  The file is named to be collected last.
"""
import pytest
import torch

from mixture_experts_layer_89_b300 import build, moe
from synth import WORKLOADS, Workload, make_inputs


def _route(wl, inp, noalloc: bool):
    cfg = moe.config_from_workload(wl, inp["x"].shape[0])
    T, E, k = cfg.T, cfg.E, cfg.k
    dev = inp["x"].device
    out = dict(idx=torch.full((T, k), -7, dtype=torch.int32, device=dev),
               w=torch.full((T, k), -1.0, dtype=torch.float32, device=dev),
               counts=torch.full((E,), -7, dtype=torch.int32, device=dev),
               losses=torch.full((2,), -1.0, dtype=torch.float32, device=dev))
    args = (cfg, inp["x"], inp["w_router"], inp.get("logit_bias"), out["idx"], out["w"], out["counts"], out["losses"])
    if noalloc:
        moe.moe_route_noalloc(*args)
    else:
        ws = moe.alloc_workspace(cfg, dev)
        moe.moe_route(*args, ws)
        assert moe.moe_read_device_status(ws) == moe.MOE_OK
    torch.cuda.synchronize()
    return {n: t.cpu() for n, t in out.items()}


def _same(a, b):
    """Both routes run the same kernels in the same launch configuration on the same inputs, so
    every output agrees bit for bit (a stale value read back from the shared array would not)."""
    for name in ("idx", "w", "counts", "losses"):
        assert torch.equal(a[name], b[name]), name


CALLS = [
    WORKLOADS["flash_bf16"].replace(name="noalloc_flash", T=4096),
    # a smaller call right after a larger one with the same E: the array still holds the larger
    # call's per-CTA partials beyond this call's blocks
    WORKLOADS["flash_bf16"].replace(name="noalloc_flash_after_large", T=100, seed=31),
    Workload("noalloc_fine_bias", T=2001, d=512, E=64, k=6, dff=64, act="swiglu", dtype="bf16", seed=31, wseed=31,
             logit_bias0=2.0),
    WORKLOADS["tiny_fp32"],
    WORKLOADS["flash_bf16"].replace(name="noalloc_flash_small", T=100, seed=32),
    # exactly at both documented limits: T = 2^20 tokens and T * E = 2^22 (accepted, not refused)
    Workload("noalloc_at_limits", T=1 << 20, d=64, E=4, k=2, dff=64, act="swiglu", dtype="bf16", seed=33, wseed=33),
]


@pytest.mark.gpu
def test_noalloc_router_matches_workspace_router_over_calls_in_a_row():
    build.build()
    for wl in CALLS:
        inp = {n: (t.to("cuda") if t is not None else None) for n, t in make_inputs(wl, "cpu").items()}
        ref = _route(wl, inp, noalloc=False)
        got = _route(wl, inp, noalloc=True)
        _same(got, ref)
        again = _route(wl, inp, noalloc=True)      # second call in a row on the same inputs
        _same(again, ref)


def test_noalloc_router_rejects_oversized_shapes_on_host():
    build.build()
    fake = 1 << 12                                  # 16-byte aligned, never dereferenced: rejected first
    for T, E in (((1 << 20) + 1, 1), ((1 << 16) + 1, 64)):
        cfg = moe.make_config(T, 64, E, 1, 64, dtype="bf16")
        st = moe.lib().moe_route_noalloc(cfg, fake, fake, None, fake, fake, fake, fake, None)
        assert st == moe.MOE_ERR_UNSUPPORTED, (T, E, st)
