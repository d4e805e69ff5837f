"""Workload shapes and the seeded input recipe for the sparse MoE FFN layer.

Recipe (identical on every device; the random streams of a CPU and a CUDA generator differ,
so a test always hands the *same* drawn tensors to both sides):

* activations: ``x = randn(T, d)`` from ``torch.Generator(device).manual_seed(seed)``, cast to
  the layer dtype with round-to-nearest-even;
* weights: one generator seeded with ``WEIGHT_SEED_BASE + wseed`` draws, in this order,
  ``w_router [E,d]``; then for each routed expert e = 0..E-1 either
  ``w_up[e] [dff,d]`` (+ ``b_up[e]``), ``w_down[e] [d,dff]`` (+ ``b_down[e]``)   (GELU experts) or
  ``w_gate[e] [dff,d]``, ``w_up[e] [dff,d]``, ``w_down[e] [d,dff]``              (SwiGLU experts);
  then for each shared expert s the same matrices into ``ws_gate/ws_up/ws_down``; then, for a
  layer with a backup expert, its matrices into ``wb_gate/wb_up/wb_down`` (biases ``bb_up``,
  ``bb_down`` as the routed experts have them).
  Each draw is ``randn * std`` (std 0.02) in fp32, then cast to the layer dtype;
* biases are zero unless ``bias_std > 0`` (only synthetic test shapes use that);
* an optional fixed router logit bias (fp32 ``[E]``) is ``(logit_bias0, 0, ..., 0)``.

Nothing here computes any part of the layer.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch

WEIGHT_SEED_BASE = 10_000


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    dff: int
    act: str                 # "gelu" (erf form) or "swiglu"
    dtype: str               # "f32" or "bf16"
    n_shared: int = 0
    bias: bool = False       # routed experts carry biases (GELU form)
    cf: float = 0.0          # capacity factor; <= 0 means dropless
    seed: int = 0            # activation seed
    wseed: int = 0           # weight seed
    logit_bias0: float = 0.0 # fixed bias added to router logit column 0
    lb_coef: float = 0.01
    z_coef: float = 0.001
    w_std: float = 0.02
    bias_std: float = 0.0
    temperature: float = 1.0 # router temperature (a routing variant; 1 = none)
    backup: bool = False     # one backup expert takes the assignments over capacity (a routing variant)
    weights8: str = "dtype"  # expert weights stored as "int8" or "e4m3" codes with row scales (quantised
                             # from the drawn weights by the library), or in the layer dtype

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS: Dict[str, Workload] = {
    # Tiny fp32 layer: Linear(64->8) router, 8 GELU experts 64->128->64 with biases, top-2.
    "tiny_fp32": Workload("tiny_fp32", T=64, d=64, E=8, k=2, dff=128, act="gelu", dtype="f32",
                          bias=True, seed=0, wseed=0),
    # 'Flash'-scale layer: 16 GELU experts 1024->4096->1024, top-2, capacity factor 1.25.
    "flash_bf16": Workload("flash_bf16", T=8192, d=1024, E=16, k=2, dff=4096, act="gelu",
                           dtype="bf16", bias=True, cf=1.25, seed=1, wseed=1),
    # Fine-grained layer: 64 routed SwiGLU experts (top-6) + 2 shared, d_ffn 1024, dropless.
    "finegrained_bf16": Workload("finegrained_bf16", T=16384, d=2048, E=64, k=6, dff=1024,
                                 act="swiglu", dtype="bf16", n_shared=2, seed=2, wseed=2),
    # Decode-shaped call on the fine-grained layer's weights: 32 tokens.
    "decode_bf16": Workload("decode_bf16", T=32, d=2048, E=64, k=6, dff=1024, act="swiglu",
                            dtype="bf16", n_shared=2, seed=3, wseed=2),
    # Large skewed layer: 128 SwiGLU experts 4096->6144->4096, top-2, +2.0 on logit 0.
    "skewed_bf16": Workload("skewed_bf16", T=16384, d=4096, E=128, k=2, dff=6144, act="swiglu",
                            dtype="bf16", seed=4, wseed=4, logit_bias0=2.0),
    "skewed_cf1_bf16": Workload("skewed_cf1_bf16", T=16384, d=4096, E=128, k=2, dff=6144,
                                act="swiglu", dtype="bf16", cf=1.0, seed=4, wseed=4,
                                logit_bias0=2.0),
    # The decode-shaped call with its experts stored as per-row scaled INT8 codes.
    "decode_int8_bf16": Workload("decode_int8_bf16", T=32, d=2048, E=64, k=6, dff=1024, act="swiglu",
                                 dtype="bf16", n_shared=2, seed=3, wseed=2, weights8="int8"),
    # The skewed layer with its experts stored as INT8 codes (9.7 GB instead of 19.3 GB).
    "skewed_int8_bf16": Workload("skewed_int8_bf16", T=16384, d=4096, E=128, k=2, dff=6144, act="swiglu",
                                 dtype="bf16", seed=4, wseed=4, logit_bias0=2.0, weights8="int8"),
    # Profiling stand-in for the skewed layer (kernel counters on a few GB of device memory): the
    # same expert shape and about the same rows per expert (~256), 16 experts instead of 128.
    "skewed_e16_bf16": Workload("skewed_e16_bf16", T=2048, d=4096, E=16, k=2, dff=6144, act="swiglu",
                                dtype="bf16", seed=5, wseed=5, logit_bias0=2.0),
}


def workload(name: str, **overrides) -> Workload:
    wl = WORKLOADS[name]
    return wl.replace(**overrides) if overrides else wl


def _draw(gen: torch.Generator, shape, std: float, dtype, device) -> torch.Tensor:
    return (torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std).to(dtype)


def make_inputs(wl: Workload, device: str = "cpu", T: Optional[int] = None) -> Dict[str, Optional[torch.Tensor]]:
    """Draw every input of the layer for workload ``wl`` on ``device`` (see module docstring)."""
    T = wl.T if T is None else T
    dt = wl.torch_dtype
    dev = torch.device(device)
    gx = torch.Generator(device=dev).manual_seed(wl.seed)
    gw = torch.Generator(device=dev).manual_seed(WEIGHT_SEED_BASE + wl.wseed)
    out: Dict[str, Optional[torch.Tensor]] = {}
    out["x"] = torch.randn((T, wl.d), generator=gx, device=dev, dtype=torch.float32).to(dt)
    out["w_router"] = _draw(gw, (wl.E, wl.d), wl.w_std, dt, dev)
    if wl.logit_bias0 != 0.0:
        lb = torch.zeros(wl.E, dtype=torch.float32, device=dev)
        lb[0] = wl.logit_bias0
        out["logit_bias"] = lb
    else:
        out["logit_bias"] = None

    E, d, f = wl.E, wl.d, wl.dff
    swiglu = wl.act == "swiglu"
    w_gate = torch.empty((E, f, d), dtype=dt, device=dev) if swiglu else None
    w_up = torch.empty((E, f, d), dtype=dt, device=dev)
    w_down = torch.empty((E, d, f), dtype=dt, device=dev)
    b_up = torch.zeros((E, f), dtype=dt, device=dev) if wl.bias else None
    b_down = torch.zeros((E, d), dtype=dt, device=dev) if wl.bias else None
    for e in range(E):
        if swiglu:
            w_gate[e] = _draw(gw, (f, d), wl.w_std, dt, dev)
        w_up[e] = _draw(gw, (f, d), wl.w_std, dt, dev)
        if wl.bias and wl.bias_std > 0:
            b_up[e] = _draw(gw, (f,), wl.bias_std, dt, dev)
        w_down[e] = _draw(gw, (d, f), wl.w_std, dt, dev)
        if wl.bias and wl.bias_std > 0:
            b_down[e] = _draw(gw, (d,), wl.bias_std, dt, dev)
    out.update(w_gate=w_gate, w_up=w_up, w_down=w_down, b_up=b_up, b_down=b_down)

    S = wl.n_shared
    if S > 0:
        ws_gate = torch.empty((S, f, d), dtype=dt, device=dev) if swiglu else None
        ws_up = torch.empty((S, f, d), dtype=dt, device=dev)
        ws_down = torch.empty((S, d, f), dtype=dt, device=dev)
        for s in range(S):
            if swiglu:
                ws_gate[s] = _draw(gw, (f, d), wl.w_std, dt, dev)
            ws_up[s] = _draw(gw, (f, d), wl.w_std, dt, dev)
            ws_down[s] = _draw(gw, (d, f), wl.w_std, dt, dev)
        out.update(ws_gate=ws_gate, ws_up=ws_up, ws_down=ws_down)
    else:
        out.update(ws_gate=None, ws_up=None, ws_down=None)
    if wl.backup:
        wb_gate = _draw(gw, (f, d), wl.w_std, dt, dev) if swiglu else None
        wb_up = _draw(gw, (f, d), wl.w_std, dt, dev)
        bb_up = (_draw(gw, (f,), wl.bias_std, dt, dev) if wl.bias_std > 0 else torch.zeros(f, dtype=dt, device=dev)) \
            if wl.bias else None
        wb_down = _draw(gw, (d, f), wl.w_std, dt, dev)
        bb_down = (_draw(gw, (d,), wl.bias_std, dt, dev) if wl.bias_std > 0 else torch.zeros(d, dtype=dt, device=dev)) \
            if wl.bias else None
        out.update(wb_gate=wb_gate, wb_up=wb_up, wb_down=wb_down, bb_up=bb_up, bb_down=bb_down)
    else:
        out.update(wb_gate=None, wb_up=None, wb_down=None, bb_up=None, bb_down=None)
    return out
