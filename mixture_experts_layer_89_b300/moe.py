"""ctypes binding of ``libmoe.so`` with the same names as the C ABI in ``include/moe.h``.

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.  PyTorch
supplies device memory and the current CUDA stream.  There is no CPU fallback: if the library
is missing or was built without a GPU-capable toolchain, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_STATUS = 0, -1, -2, -3, -4, -5
MOE_F32, MOE_BF16 = 0, 1
MOE_ACT_GELU_ERF, MOE_ACT_SWIGLU = 0, 1

_c_i32 = ctypes.c_int32
_c_p = ctypes.c_void_p


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", _c_i32), ("d", _c_i32), ("E", _c_i32), ("k", _c_i32), ("dff", _c_i32),
                ("n_shared", _c_i32), ("act", _c_i32), ("dtype", _c_i32), ("has_bias", _c_i32),
                ("capacity_factor", ctypes.c_float), ("lb_coef", ctypes.c_float), ("z_coef", ctypes.c_float),
                ("router_temperature", ctypes.c_float), ("backup_expert", _c_i32), ("expert_weights", _c_i32)]


class MoeWeights(ctypes.Structure):
    _fields_ = [("w_router", _c_p), ("router_logit_bias", _c_p), ("w_up", _c_p), ("w_gate", _c_p),
                ("w_down", _c_p), ("b_up", _c_p), ("b_down", _c_p), ("ws_up", _c_p), ("ws_gate", _c_p),
                ("ws_down", _c_p), ("wb_up", _c_p), ("wb_gate", _c_p), ("wb_down", _c_p), ("bb_up", _c_p),
                ("bb_down", _c_p), ("s_up", _c_p), ("s_gate", _c_p), ("s_down", _c_p), ("ss_up", _c_p),
                ("ss_gate", _c_p), ("ss_down", _c_p), ("sb_up", _c_p), ("sb_gate", _c_p), ("sb_down", _c_p)]


class MoeForwardViews(ctypes.Structure):
    _fields_ = [("topk_idx", _c_p), ("topk_w", _c_p), ("counts", _c_p), ("offsets", _c_p), ("row_of", _c_p),
                ("tok_of", _c_p), ("x_perm", _c_p), ("y_perm", _c_p)]


class MoeExpertGrads(ctypes.Structure):
    _fields_ = [("dw_up", _c_p), ("dw_gate", _c_p), ("dw_down", _c_p), ("db_up", _c_p), ("db_down", _c_p),
                ("dws_up", _c_p), ("dws_gate", _c_p), ("dws_down", _c_p)]


# expert weight storage (moe_expert_weights)
EXPERT_WEIGHTS = {"dtype": 0, "int8": 1, "e4m3": 2}


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        detail = ""
        if status == MOE_ERR_CUDA:
            msg = lib().moe_last_error().decode()
            detail = f" [{msg}]" if msg else ""
        super().__init__(f"{where}: {moe_status_string(status)} ({status}){detail}")
        self.status = status


_LIB: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """Load libmoe.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m mixture_experts_layer_89_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER
        cfgp = P(MoeConfig)
        L.moe_workspace_size.argtypes = [cfgp, P(ctypes.c_size_t)]
        L.moe_capacity.argtypes = [cfgp, P(_c_i32), P(_c_i32)]
        L.moe_route.argtypes = [cfgp, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p]
        L.moe_route_noalloc.argtypes = [cfgp, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p]
        L.moe_permute.argtypes = [cfgp, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p]
        L.moe_expert_ffn.argtypes = [cfgp, _c_p, _c_p, P(MoeWeights), _c_p, _c_p, _c_p, _c_p, _c_p]
        L.moe_combine.argtypes = [cfgp, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p]
        L.moe_layer_forward.argtypes = [cfgp, P(MoeWeights), _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p]
        L.moe_layer_forward_timed.argtypes = [cfgp, P(MoeWeights), _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p,
                                              P(_c_p), _c_i32]
        L.moe_read_device_status.argtypes = [_c_p, _c_p]
        L.moe_layer_forward_launches.argtypes = [cfgp]
        L.moe_set_wait_limit.argtypes = [_c_p, ctypes.c_uint64, _c_p]
        L.moe_route_diagnostics.argtypes = [cfgp, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p]
        L.moe_route_stats.argtypes = [cfgp, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p]
        L.moe_quantize_experts.argtypes = [_c_p, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_p, _c_p, _c_p, _c_p]
        L.moe_combine_backward.argtypes = [cfgp, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p]
        L.moe_route_backward.argtypes = [cfgp, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, ctypes.c_float,
                                         ctypes.c_float, _c_p, _c_p, _c_p, _c_p, _c_p]
        L.moe_route_backward_scratch_size.argtypes = [cfgp, P(ctypes.c_size_t)]
        L.moe_expert_backward_scratch_size.argtypes = [cfgp, P(ctypes.c_size_t)]
        L.moe_workspace_views.argtypes = [cfgp, _c_p, P(MoeForwardViews)]
        L.moe_expert_ffn_backward.argtypes = [cfgp, P(MoeWeights), _c_p, _c_p, _c_p, _c_p, _c_p, _c_p,
                                              P(MoeExpertGrads), _c_p, _c_p, _c_p]
        L.moe_status_string.argtypes = [_c_i32]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_last_error.argtypes = []
        L.moe_last_error.restype = ctypes.c_char_p
        for name in ("moe_workspace_size", "moe_capacity", "moe_route", "moe_route_noalloc", "moe_permute",
                     "moe_expert_ffn", "moe_combine", "moe_layer_forward", "moe_layer_forward_timed",
                     "moe_read_device_status", "moe_layer_forward_launches", "moe_route_stats",
                     "moe_set_wait_limit", "moe_route_diagnostics", "moe_quantize_experts", "moe_combine_backward",
                     "moe_route_backward", "moe_route_backward_scratch_size", "moe_expert_backward_scratch_size",
                     "moe_expert_ffn_backward", "moe_workspace_views"):
            getattr(L, name).restype = _c_i32
        _LIB = L
    return _LIB


EXPORTED = ("moe_workspace_size", "moe_capacity", "moe_route", "moe_route_noalloc", "moe_permute", "moe_expert_ffn",
            "moe_combine", "moe_layer_forward", "moe_layer_forward_timed", "moe_read_device_status",
            "moe_layer_forward_launches", "moe_route_stats", "moe_set_wait_limit", "moe_route_diagnostics",
            "moe_quantize_experts", "moe_combine_backward", "moe_route_backward", "moe_route_backward_scratch_size",
            "moe_expert_backward_scratch_size", "moe_expert_ffn_backward", "moe_workspace_views", "moe_status_string",
            "moe_last_error")


# ----------------------------------------------------------------------------- marshalling
def _p(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _s(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def make_config(T: int, d: int, E: int, k: int, dff: int, act: str = "gelu", dtype: str = "bf16",
                n_shared: int = 0, has_bias: bool = False, capacity_factor: float = 0.0,
                lb_coef: float = 0.01, z_coef: float = 0.001, temperature: float = 1.0,
                backup_expert: bool = False, expert_weights: str = "dtype") -> MoeConfig:
    return MoeConfig(T, d, E, k, dff, n_shared, MOE_ACT_SWIGLU if act == "swiglu" else MOE_ACT_GELU_ERF,
                     MOE_BF16 if dtype == "bf16" else MOE_F32, int(bool(has_bias)), float(capacity_factor),
                     float(lb_coef), float(z_coef), float(temperature), int(bool(backup_expert)),
                     EXPERT_WEIGHTS[expert_weights])


def config_from_workload(wl, T: Optional[int] = None) -> MoeConfig:
    return make_config(wl.T if T is None else T, wl.d, wl.E, wl.k, wl.dff, wl.act, wl.dtype, wl.n_shared,
                       wl.bias, wl.cf, wl.lb_coef, wl.z_coef, getattr(wl, "temperature", 1.0),
                       getattr(wl, "backup", False), getattr(wl, "weights8", "dtype"))


def make_weights(t: Dict[str, Optional[torch.Tensor]]) -> MoeWeights:
    """MoeWeights over the tensors of ``t`` (keys as produced by ``synth.make_inputs``)."""
    w = MoeWeights(*[_p(t.get(n)) for n in ("w_router", "logit_bias", "w_up", "w_gate", "w_down", "b_up", "b_down",
                                            "ws_up", "ws_gate", "ws_down", "wb_up", "wb_gate", "wb_down", "bb_up",
                                            "bb_down", "s_up", "s_gate", "s_down", "ss_up", "ss_gate", "ss_down",
                                            "sb_up", "sb_gate", "sb_down")])
    w._keep = t  # keep the tensors alive as long as the struct
    return w


# ----------------------------------------------------------------------------- C ABI, same names
def moe_status_string(s: int) -> str:
    return lib().moe_status_string(int(s)).decode()


def moe_workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_size")
    return int(n.value)


def moe_capacity(cfg: MoeConfig):
    cap, amax = _c_i32(0), _c_i32(0)
    _check(lib().moe_capacity(ctypes.byref(cfg), ctypes.byref(cap), ctypes.byref(amax)), "moe_capacity")
    return int(cap.value), int(amax.value)


def moe_route(cfg, x, w_router, logit_bias, topk_idx, topk_w, counts, losses, ws, stream=None):
    _check(lib().moe_route(ctypes.byref(cfg), _p(x), _p(w_router), _p(logit_bias), _p(topk_idx), _p(topk_w),
                           _p(counts), _p(losses), _p(ws), _s(stream)), "moe_route")


def moe_route_noalloc(cfg, x, w_router, logit_bias, topk_idx, topk_w, counts, losses, stream=None):
    """moe_route without a workspace: the library's fixed device scratch array is used instead."""
    _check(lib().moe_route_noalloc(ctypes.byref(cfg), _p(x), _p(w_router), _p(logit_bias), _p(topk_idx),
                                   _p(topk_w), _p(counts), _p(losses), _s(stream)), "moe_route_noalloc")


def moe_permute(cfg, x, topk_idx, counts, offsets, kept, row_of, tok_of, x_perm, ws, stream=None):
    _check(lib().moe_permute(ctypes.byref(cfg), _p(x), _p(topk_idx), _p(counts), _p(offsets), _p(kept),
                             _p(row_of), _p(tok_of), _p(x_perm), _p(ws), _s(stream)), "moe_permute")


def moe_expert_ffn(cfg, x_perm, offsets, weights: MoeWeights, y_perm, x, y_shared, ws, stream=None):
    _check(lib().moe_expert_ffn(ctypes.byref(cfg), _p(x_perm), _p(offsets), ctypes.byref(weights), _p(y_perm),
                                _p(x), _p(y_shared), _p(ws), _s(stream)), "moe_expert_ffn")


def moe_combine(cfg, y_perm, row_of, topk_w, y_shared, y, stream=None):
    _check(lib().moe_combine(ctypes.byref(cfg), _p(y_perm), _p(row_of), _p(topk_w), _p(y_shared), _p(y),
                             _s(stream)), "moe_combine")


def moe_layer_forward(cfg, weights: MoeWeights, x, y, losses, counts_out, drops_out, ws, stream=None):
    _check(lib().moe_layer_forward(ctypes.byref(cfg), ctypes.byref(weights), _p(x), _p(y), _p(losses),
                                   _p(counts_out), _p(drops_out), _p(ws), _s(stream)), "moe_layer_forward")


def moe_layer_forward_timed(cfg, weights: MoeWeights, x, y, losses, counts_out, drops_out, ws,
                            events: Sequence[torch.cuda.Event], stream=None):
    handles = [ev.cuda_event for ev in events]
    if not all(handles):
        raise ValueError("events must have been recorded once (torch creates them lazily)")
    arr = (_c_p * len(events))(*handles)
    _check(lib().moe_layer_forward_timed(ctypes.byref(cfg), ctypes.byref(weights), _p(x), _p(y), _p(losses),
                                         _p(counts_out), _p(drops_out), _p(ws), _s(stream), arr, len(events)),
           "moe_layer_forward_timed")


def moe_read_device_status(ws, stream=None) -> int:
    """Synchronise and return (and clear) the device status word of ``ws`` as a status code."""
    return int(lib().moe_read_device_status(_p(ws), _s(stream)))


def moe_route_stats(cfg, topk_idx, offsets, coact, stats, ws, stream=None):
    _check(lib().moe_route_stats(ctypes.byref(cfg), _p(topk_idx), _p(offsets), _p(coact), _p(stats), _p(ws),
                                 _s(stream)), "moe_route_stats")


def moe_set_wait_limit(ws, limit_ns: int, stream=None):
    """Shorten (or, with 0, restore) the router's bounded waits for calls that use ``ws``."""
    _check(lib().moe_set_wait_limit(_p(ws), int(limit_ns), _s(stream)), "moe_set_wait_limit")


def moe_route_diagnostics(cfg, x, w_router, logit_bias, diag, entropy_tok, ws, stream=None):
    _check(lib().moe_route_diagnostics(ctypes.byref(cfg), _p(x), _p(w_router), _p(logit_bias), _p(diag),
                                       _p(entropy_tok), _p(ws), _s(stream)), "moe_route_diagnostics")


def moe_layer_forward_launches(cfg) -> int:
    return int(lib().moe_layer_forward_launches(ctypes.byref(cfg)))


def moe_quantize_experts(w, fmt: str, blocks: int, rows: int, cols: int, codes, scale, nonfinite=None,
                         stream=None):
    """Per-row scaled 8-bit codes of ``w`` [blocks, rows, cols] (``fmt`` "int8" or "e4m3")."""
    dtype = MOE_BF16 if w.dtype == torch.bfloat16 else MOE_F32
    _check(lib().moe_quantize_experts(_p(w), dtype, EXPERT_WEIGHTS[fmt], int(blocks), int(rows), int(cols),
                                      _p(codes), _p(scale), _p(nonfinite), _s(stream)), "moe_quantize_experts")


def moe_combine_backward(cfg, dy, y_perm, row_of, topk_w, dw, dy_perm, stream=None):
    _check(lib().moe_combine_backward(ctypes.byref(cfg), _p(dy), _p(y_perm), _p(row_of), _p(topk_w), _p(dw),
                                      _p(dy_perm), _s(stream)), "moe_combine_backward")


def moe_route_backward_scratch_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_route_backward_scratch_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_route_backward_scratch_size")
    return int(n.value)


def moe_route_backward(cfg, x, w_router, logit_bias, topk_idx, topk_w, counts, dw, dlb, dzl, dz, dw_router, dx,
                       scratch=None, stream=None):
    _check(lib().moe_route_backward(ctypes.byref(cfg), _p(x), _p(w_router), _p(logit_bias), _p(topk_idx),
                                    _p(topk_w), _p(counts), _p(dw), float(dlb), float(dzl), _p(dz), _p(dw_router),
                                    _p(dx), _p(scratch), _s(stream)), "moe_route_backward")


def moe_workspace_views(cfg: MoeConfig, ws) -> Dict[str, int]:
    """Device addresses of the forward's intermediates inside workspace ``ws`` (see moe.h)."""
    v = MoeForwardViews()
    _check(lib().moe_workspace_views(ctypes.byref(cfg), _p(ws), ctypes.byref(v)), "moe_workspace_views")
    return {name: getattr(v, name) for name, _ in MoeForwardViews._fields_}


def moe_expert_backward_scratch_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_expert_backward_scratch_size(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_expert_backward_scratch_size")
    return int(n.value)


def make_expert_grads(g: Dict[str, Optional[torch.Tensor]]) -> MoeExpertGrads:
    """MoeExpertGrads over the fp32 tensors of ``g`` (keys dw_up, dw_gate, dw_down, db_up, db_down,
    dws_up, dws_gate, dws_down; missing keys are NULL)."""
    s = MoeExpertGrads(*[_p(g.get(n)) for n in ("dw_up", "dw_gate", "dw_down", "db_up", "db_down", "dws_up",
                                                "dws_gate", "dws_down")])
    s._keep = g
    return s


def moe_expert_ffn_backward(cfg, weights: MoeWeights, x, x_perm, offsets, row_of, dy, dy_perm,
                            grads: MoeExpertGrads, dx, scratch, stream=None):
    _check(lib().moe_expert_ffn_backward(ctypes.byref(cfg), ctypes.byref(weights), _p(x), _p(x_perm), _p(offsets),
                                         _p(row_of), _p(dy), _p(dy_perm), ctypes.byref(grads), _p(dx),
                                         _p(scratch), _s(stream)), "moe_expert_ffn_backward")


# ----------------------------------------------------------------------------- convenience
_QUANT_KEYS = (("w_up", "s_up", False), ("w_gate", "s_gate", False), ("w_down", "s_down", False),
               ("ws_up", "ss_up", False), ("ws_gate", "ss_gate", False), ("ws_down", "ss_down", True),
               ("wb_up", "sb_up", False), ("wb_gate", "sb_gate", False), ("wb_down", "sb_down", False))


def quantize_expert_tensors(t: Dict[str, Optional[torch.Tensor]], fmt: str, stream=None):
    """A copy of the layer tensors ``t`` whose expert matrices are replaced by 8-bit codes (int8 or
    uint8 E4M3 tensors of the same shapes) with their row scales under the s_* / ss_* / sb_* keys,
    quantised on the GPU by moe_quantize_experts (the shared experts' down matrices share one scale
    per row).  Raises if a weight is not finite."""
    out = dict(t)
    bad = torch.zeros(1, dtype=torch.int32, device=next(v for v in t.values() if v is not None).device)
    for wk, sk, joint in _QUANT_KEYS:
        w = t.get(wk)
        if w is None:
            continue
        w3 = w.reshape(1, *w.shape) if w.dim() == 2 else w
        B, R, C = w3.shape
        codes = torch.empty(w3.shape, dtype=torch.int8 if fmt == "int8" else torch.uint8, device=w.device)
        blocks, rows = (B, R) if joint else (1, B * R)
        scale = torch.empty(rows, dtype=torch.float32, device=w.device)
        moe_quantize_experts(w3, fmt, blocks, rows, C, codes, scale, bad, stream)
        out[wk] = codes.reshape(w.shape)
        out[sk] = scale if joint else scale.reshape(w.shape[:-1])
    if int(bad.item()):
        raise ValueError(f"{int(bad.item())} non-finite expert weights")
    return out
def alloc_workspace(cfg: MoeConfig, device="cuda") -> torch.Tensor:
    """Zero-filled workspace (the status word must start at zero)."""
    return torch.zeros(max(moe_workspace_size(cfg), 256), dtype=torch.uint8, device=device)


class MoELayer:
    """Holds a config, the weights and a workspace; ``forward(x)`` runs ``moe_layer_forward``."""

    def __init__(self, cfg: MoeConfig, tensors: Dict[str, Optional[torch.Tensor]], device="cuda"):
        self.cfg = cfg
        self.weights = make_weights(tensors)
        self.ws = alloc_workspace(cfg, device)
        self.device = device

    def forward(self, x: torch.Tensor, stream=None):
        c = self.cfg
        y = torch.empty_like(x)
        losses = torch.empty(2, dtype=torch.float32, device=x.device)
        counts = torch.empty(c.E, dtype=torch.int32, device=x.device)
        drops = torch.empty(1, dtype=torch.int32, device=x.device)
        moe_layer_forward(c, self.weights, x, y, losses, counts, drops, self.ws, stream)
        return y, losses, counts, drops
