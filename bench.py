"""Benchmark of the sparse MoE FFN layer forward on B300 (one JSON line on stdout, rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one full ``moe_layer_forward`` (route, dispatch, expert FFNs, combine, losses) over one
batch of synthetic tokens already resident in HBM.  Per-GPU work is fixed (``"scaling": "weak"``):
under torchrun every rank runs an independent replica of the layer on its own GPU (the layer
needs no exchange between replicas), and the value counts the tokens of all ranks over the
slowest rank's time.

``--impl reference`` times the CPU oracle (fp64 NumPy, explicit per-expert loop) on a bounded
token sample of the same workload; only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from synth import WORKLOADS, make_inputs  # noqa: E402

DEFAULT_WORKLOAD = "skewed_bf16"
# the other workloads, each measured as a sub-record of the single-GPU line
SUB_WORKLOADS = ("tiny_fp32", "flash_bf16", "finegrained_bf16", "decode_bf16", "decode_int8_bf16", "skewed_bf16",
                 "skewed_cf1_bf16")
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the up-projection
# kernel, from ncu captures (profiles/k_proj_tc_skewed_e16_bf16.md), keyed by workload; valid only
# while gemm_tc.cu and common.cuh hash to src_sha1.  skewed_e16_bf16 is measured; skewed_bf16 is
# too large to capture under a full metric set, so its figure is the stand-in's traffic per
# algorithmic byte (1.0143) times the full launch's algorithmic bytes (weights of 128 experts,
# token rows in, hidden rows out).
NCU_TRAFFIC = {
    "skewed_e16_bf16": {"bytes": 1669249536 + 49530112, "src_sha1": "4289058b31e7b631343f91ba81d028ca6d3e9552"},
    "skewed_bf16": {"bytes": 13750237184, "src_sha1": "4289058b31e7b631343f91ba81d028ca6d3e9552",
                    "scaled_from": "skewed_e16_bf16"},
}


METRIC = "MoE-layer fwd tokens/s and expert-GEMM TFLOP/s (% of bf16 peak) on 1 B300"
L2_BYTES = 128 * 1024 * 1024  # B300 L2 is 126 MB; flush by writing twice this


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_src_sha1():
    h = hashlib.sha1()
    for name in ("gemm_tc.cu", "common.cuh"):
        with open(os.path.join(ROOT, "mixture_experts_layer_89_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


class _Nvml:
    """Minimal read-only NVML access through ctypes (libnvidia-ml ships with the driver)."""

    SM = 1  # NVML_CLOCK_SM
    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, torch_device: int):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.h = ctypes.c_void_p()
        p = torch.cuda.get_device_properties(torch_device)
        bus = ("%08x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)).encode()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(self.h)) != 0:
            raise RuntimeError(f"no NVML handle for PCI bus {bus.decode()}")
        self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def _u32(self, fn, *args):
        v = self.c.c_uint(0)
        if fn(self.h, *args, self.c.byref(v)) != 0:
            raise RuntimeError(fn.__name__)
        return v.value

    def sample(self):
        r = self.c.c_ulonglong(0)
        if self._reasons(self.h, self.c.byref(r)) != 0:
            raise RuntimeError("clock event reasons")
        return (self._u32(self.lib.nvmlDeviceGetClockInfo, self.SM), self._u32(self.lib.nvmlDeviceGetPowerUsage) / 1e3,
                r.value)

    def max_sm(self):
        return self._u32(self.lib.nvmlDeviceGetMaxClockInfo, self.SM)

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """Samples the SM clock, power and clock-event (throttle) reasons through NVML (read-only
    queries) every ~1 ms in a background thread while the timed region runs."""

    def __init__(self, torch_device: int):
        self.dev = torch_device
        self.rows = []
        self.err = None
        self.nv = None

    def _run(self):
        while not self.stop.is_set():
            try:
                self.rows.append(self.nv.sample())
            except Exception as e:  # pragma: no cover
                self.err = str(e)
                return
            time.sleep(0.001)

    def __enter__(self):
        import threading
        try:
            self.nv = _Nvml(self.dev)
            self.smax = self.nv.max_sm()
            self.stop = threading.Event()
            self.th = threading.Thread(target=self._run, daemon=True)
            self.th.start()
            time.sleep(0.01)  # first samples before the timed work starts
        except Exception as e:
            self.nv = None
            self.err = str(e)
        return self

    def __exit__(self, *exc):
        if self.nv is not None:
            self.stop.set()
            self.th.join(timeout=5)
            self.nv.close()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [f"no samples ({self.err})"]}
        reasons = sorted({n for n, bit in _Nvml.REASONS.items() for r in self.rows if r[2] & bit})
        return {"sm_mhz": statistics.median(r[0] for r in self.rows), "sm_max_mhz": self.smax,
                "reasons": reasons, "samples": len(self.rows), "power_w_max": round(max(r[1] for r in self.rows), 1),
                "source": "NVML (libnvidia-ml via ctypes), ~1 ms period, timed region only"}


def weight_elt(wl) -> int:
    """Bytes per expert weight: 1 for 8-bit codes, else the layer dtype's."""
    return 1 if getattr(wl, "weights8", "dtype") != "dtype" else (2 if wl.dtype == "bf16" else 4)


def weight_bytes_of(wl) -> int:
    """Expert weights (routed and shared) one layer pass streams."""
    return (wl.E + wl.n_shared) * (3 if wl.act == "swiglu" else 2) * wl.d * wl.dff * weight_elt(wl)


def flushes_l2(wl) -> bool:
    """Workloads whose weights are under twice the L2 get an L2 flush before every timed step."""
    return weight_bytes_of(wl) < 2 * L2_BYTES


def arm_config(wl, ws_n: int) -> dict:
    """The workload the line is quoted on (both arms print the same one)."""
    w8 = {} if getattr(wl, "weights8", "dtype") == "dtype" else {
        "expert_weights": f"{wl.weights8} codes + fp32 row scales (quantised once, before timing)"}
    return {**w8, "workload": wl.name, "T": wl.T, "d_model": wl.d, "experts": wl.E, "top_k": wl.k,
            "d_ffn": wl.dff, "act": wl.act, "shared_experts": wl.n_shared,
            "capacity_factor": wl.cf if wl.cf > 0 else None,
            "parallelism": f"replicas x{ws_n} (no collective)",
            "timing": "CUDA-graph replay of one moe_layer_forward per step",
            "l2": ("L2 flushed before every timed step (256 MB write outside the events)" if flushes_l2(wl) else
                   "inputs larger than L2 (expert weights %.0f MB per step)" % (weight_bytes_of(wl) / 1e6))}


def expert_flops(wl, kept_rows: int, T: int):
    """Algorithmic expert FLOPs: 2 * rows * (matrices * d * dff) for the kept routed rows plus the
    shared experts on every token; (up, down) split."""
    m_up = 2 if wl.act == "swiglu" else 1
    up = 2.0 * kept_rows * m_up * wl.d * wl.dff
    down = 2.0 * kept_rows * wl.d * wl.dff
    sh_up = 2.0 * T * wl.n_shared * m_up * wl.d * wl.dff
    sh_down = 2.0 * T * wl.n_shared * wl.d * wl.dff
    return up, down, sh_up, sh_down


# ------------------------------------------------------------------------------ our arm
def measure(args, wl, ws_n, local, full: bool, cpu_flops: float = 0.0):
    """Time one workload on this rank's GPU.  ``full`` adds the headline-only parts (eager timing,
    routing statistics, the end-to-end run with host buffers, launch count); ``cpu_flops`` > 0 adds
    a CPU-oracle leg on a bounded token sample of the same (device-drawn) tensors, copied to host
    memory before its timer starts."""
    from mixture_experts_layer_89_b300 import moe

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = make_inputs(wl, str(dev))
    if getattr(wl, "weights8", "dtype") != "dtype":  # 8-bit experts: quantised once, by the library
        inp = moe.quantize_expert_tensors(inp, wl.weights8)
    cfg = moe.config_from_workload(wl)
    layer = moe.MoELayer(cfg, inp, device=dev)
    T, d = wl.T, wl.d
    y = torch.empty_like(inp["x"])
    losses = torch.empty(2, dtype=torch.float32, device=dev)
    counts = torch.empty(wl.E, dtype=torch.int32, device=dev)
    drops = torch.empty(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    n_ev = 7
    n_stage_steps = min(args.steps, 20)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(n_stage_steps)]
    for row in evs:          # torch creates the CUDA event on first record: make the handles exist
        for ev in row:
            ev.record(stream)
    torch.cuda.synchronize(dev)

    def step(i=None, s=stream):
        if i is None:
            moe.moe_layer_forward(cfg, layer.weights, inp["x"], y, losses, counts, drops, layer.ws, s)
        else:
            moe.moe_layer_forward_timed(cfg, layer.weights, inp["x"], y, losses, counts, drops, layer.ws, evs[i], s)

    for _ in range(args.warmup):
        step()
    st = moe.moe_read_device_status(layer.ws)
    if st != 0:
        raise RuntimeError(f"{wl.name}: device status after warm-up: {moe.moe_status_string(st)}")
    kept_rows = int(wl.T * wl.k - drops.item())

    # one layer pass captured as a CUDA graph: the replay issues the same kernels with no host work
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(s=torch.cuda.current_stream(dev))
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize(dev)

    # weights the step streams; below twice the L2 size the L2 is flushed (a 256 MB write outside
    # the timed events) before every timed step instead
    elt = 2 if wl.dtype == "bf16" else 4
    welt = weight_elt(wl)
    # 8-bit experts also read one fp32 scale per weight row
    srow = 4.0 / wl.d if welt == 1 else 0.0
    srow_dn = 4.0 / wl.dff if welt == 1 else 0.0
    flush_l2 = flushes_l2(wl)
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush_l2 else None

    def timed(fn, n):
        if flush_l2:
            return timed_flushed(fn, n)
        barrier()
        torch.cuda.synchronize(dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(n):
            fn(i)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        return max_over_ranks(t0.elapsed_time(t1)) / n

    def timed_flushed(fn, n):
        barrier()
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            flush_buf.fill_(i & 0xff)
            ev[i][0].record(stream)
            fn(i)
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        return max_over_ranks(sum(a.elapsed_time(b) for a, b in ev)) / n

    # stage times first (right after the warm-up, so that they see the same clocks as the steps
    # that follow on a power-limited part), then the graph-replayed steps, then the eager ones
    with ClockSampler(local) as clk_stages:
        timed(lambda i: step(i), n_stage_steps)
    with ClockSampler(local) as clk:
        ms_step = timed(lambda i: graph.replay(), args.steps)
    ms_eager = timed(lambda i: step(), args.steps) if full else None
    st = moe.moe_read_device_status(layer.ws)
    if st != 0:
        raise RuntimeError(f"{wl.name}: device status after timing: {moe.moe_status_string(st)}")
    stages = ["route", "dispatch", "up", "down", "shared", "combine"]
    stage_ms = {s: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n_stage_steps))
                for j, s in enumerate(stages)}

    up, down, sh_up, sh_down = expert_flops(wl, kept_rows, T)
    total_expert = up + down + sh_up + sh_down
    peaks, peak_src = load_peaks()
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    clocks = clk.summary()
    stage_clk = clk_stages.summary()
    # the burst peak for a kernel in a short step; the sustained (power-capped) one when the region
    # the stage times come from ran under the power cap with the SM clock held below its maximum
    smax = stage_clk.get("sm_max_mhz") or 0
    capped = ("sw_power_cap" in (stage_clk.get("reasons") or []) and smax > 0
              and (stage_clk.get("sm_mhz") or smax) < 0.95 * smax)
    peak, peak_name = (peak_sus, "bf16_tflops_sustained") if capped else (peak_burst, "bf16_tflops")
    traffic, traffic_note = None, None
    rec = NCU_TRAFFIC.get(wl.name)
    if rec and rec.get("src_sha1") == kernel_src_sha1():
        traffic = rec["bytes"]
        traffic_note = ("scaled from the ncu capture of " + rec["scaled_from"]) if rec.get("scaled_from") else "ncu capture"
    touched = int((counts > 0).sum().item())
    m_up = 2 if wl.act == "swiglu" else 1
    expert_ms = stage_ms["up"] + stage_ms["down"] + stage_ms["shared"]
    if wl.dtype == "bf16":
        # the up-projection launch carries the routed and the shared experts' up-projections
        up_all = up + sh_up
        up_tflops = up_all / (stage_ms["up"] * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": "k_proj_tc up-projection (routed + shared experts, GELU or SwiGLU)",
                    "achieved": round(up_tflops, 2), "peak": peak, "unit": "TFLOP/s",
                    "frac": round(up_tflops / peak, 4), "frac_of_burst_peak": round(up_tflops / peak_burst, 4),
                    "frac_of_sustained_peak": round(up_tflops / peak_sus, 4),
                    "peak_source": f"{peak_src} {peak_name}", "traffic": traffic, "traffic_source": traffic_note,
                    "algorithmic_flops_per_launch": up_all}
        up_bytes = int((touched + wl.n_shared) * m_up * wl.d * wl.dff * (welt + srow)
                    + (kept_rows + (T if wl.n_shared else 0)) * wl.d * elt
                    + (kept_rows + T * wl.n_shared) * wl.dff * elt)
        if up_all / up_bytes < peak * 1e12 / (hbm * 1e9):
            # below the ridge point (few rows per expert): the up-projection streams its weights
            up_gbs = up_bytes / (stage_ms["up"] * 1e-3) / 1e9
            roofline = {"bound": "hbm", "kernel": "k_proj_tc up-projection (weight streaming)",
                        "achieved": round(up_gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(up_gbs / hbm, 4),
                        "peak_source": f"{peak_src} hbm_gbs", "traffic": traffic, "traffic_source": traffic_note,
                        "algorithmic_bytes_per_launch": up_bytes,
                        "units": f"{touched} routed + {wl.n_shared} shared experts' up weights"
                                 + (f" ({welt}-byte codes + row scales)" if welt == 1 else "")
                                 + ", token rows read, hidden rows written"}
    else:
        roofline = {"bound": "latency", "kernel": "whole fp32 layer (CUDA cores; the fp32 parity bound rules "
                    "out the tensor cores)", "achieved": round(ms_step * 1e3, 2), "unit": "us per layer",
                    "peak": None, "frac": None, "traffic": None}
    # bytes the step must move: the weights of every expert that received a token, the shared
    # experts, the router weights, x in and y out
    layer_bytes = int((touched + wl.n_shared) * wl.d * wl.dff * (m_up * (welt + srow) + welt + srow_dn)
                      + wl.E * wl.d * elt + 2 * T * wl.d * elt)
    layer_gbs = layer_bytes / (ms_step * 1e-3) / 1e9
    res = {
        "workload": wl.name,
        "value": round(job_tokens_per_s(T, ws_n, ms_step), 1), "unit": "tokens/s",
        "ms_per_step": round(ms_step, 5),
        "expert_tflops": round(total_expert / (expert_ms * 1e-3) / 1e12, 2),
        "expert_frac_of_burst_peak": round(total_expert / (expert_ms * 1e-3) / 1e12 / peak_burst, 4),
        "expert_frac_of_sustained_peak": round(total_expert / (expert_ms * 1e-3) / 1e12 / peak_sus, 4),
        "stage_ms": {k: round(v, 5) for k, v in stage_ms.items()},
        "kept_rows": kept_rows, "drops": int(wl.T * wl.k - kept_rows),
        "roofline": roofline,
        "weight_stream": {"bytes_per_step": layer_bytes, "experts_touched": touched, "GB/s": round(layer_gbs, 1),
                          "frac_of_hbm": round(layer_gbs / hbm, 4)},
        "l2": arm_config(wl, ws_n)["l2"],
        "clocks": clocks,
        "stage_clocks": {k: v for k, v in stage_clk.items() if k in ("sm_mhz", "reasons", "samples")},
    }
    if full:
        res["eager"] = {"value": round(T * ws_n / (ms_eager * 1e-3), 1), "ms_per_step": round(ms_eager, 5),
                        "note": "moe_layer_forward issued from Python every step (host launch cost included)"}
        res["route_stats"] = route_stats_of(moe, wl, cfg, inp, layer, drops, dev, stream)
        res["backward"] = backward_of(moe, wl, cfg, inp, dev, stream)
        res["e2e"] = e2e_of(moe, args, wl, cfg, inp, layer, y, counts, drops, dev, stream, ws_n)
        res["gpu_launches"] = moe.moe_layer_forward_launches(cfg) * args.steps
    del graph
    if cpu_flops > 0:
        n = cpu_sample_tokens(wl, cpu_flops)
        host = {k: (v[:n] if k == "x" else v).to("cpu") if v is not None else None for k, v in inp.items()}
        del inp, layer
        torch.cuda.empty_cache()
        res["cpu_baseline"] = cpu_leg(wl, host, n)
    else:
        del inp, layer
        torch.cuda.empty_cache()
    return res


def backward_of(moe, wl, cfg, inp, dev, stream, n=5):
    """The backward pass on this workload: moe_combine_backward, moe_route_backward and
    moe_expert_ffn_backward on the forward steps' own outputs (routing, rows, y_perm), each timed
    alone with CUDA events (n calls after two warm-ups), outside the layer's figures."""
    T, d, E, k, f, S = wl.T, wl.d, wl.E, wl.k, wl.dff, wl.n_shared
    cap, amax = moe.moe_capacity(cfg)
    ws = moe.alloc_workspace(cfg, dev)
    i32 = dict(dtype=torch.int32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    idx, tw = torch.empty((T, k), **i32), torch.empty((T, k), **f32)
    counts, losses = torch.empty(E, **i32), torch.empty(2, **f32)
    moe.moe_route(cfg, inp["x"], inp["w_router"], inp.get("logit_bias"), idx, tw, counts, losses, ws, stream)
    offsets, kept, row_of = torch.empty(E + 1, **i32), torch.empty(E, **i32), torch.empty((T, k), **i32)
    tok_of = torch.empty(max(amax, 1), **i32)
    x_perm = torch.empty((max(amax, 1), d), dtype=inp["x"].dtype, device=dev)
    moe.moe_permute(cfg, inp["x"], idx, counts, offsets, kept, row_of, tok_of, x_perm, ws, stream)
    y_perm = torch.empty((max(amax, 1), d), **f32)
    y_sh = torch.empty((T, d), **f32) if S else None
    weights = moe.make_weights(inp)
    moe.moe_expert_ffn(cfg, x_perm, offsets, weights, y_perm, inp["x"], y_sh, ws, stream)
    g = torch.Generator(device=dev).manual_seed(12345)
    dy = torch.randn((T, d), generator=g, device=dev).to(inp["x"].dtype)
    dw = torch.empty((T, k), **f32)
    dy_perm = torch.empty_like(x_perm)
    dz = torch.empty((T, E), **f32)
    dwr = torch.empty((E, d), **f32)
    dx = torch.empty((T, d), **f32)
    glu = wl.act == "swiglu"
    grads = {"dw_up": torch.empty((E, f, d), **f32), "dw_down": torch.empty((E, d, f), **f32)}
    if glu:
        grads["dw_gate"] = torch.empty((E, f, d), **f32)
    if wl.bias:
        grads["db_up"], grads["db_down"] = torch.empty((E, f), **f32), torch.empty((E, d), **f32)
    if S:
        grads["dws_up"], grads["dws_down"] = torch.empty((S, f, d), **f32), torch.empty((S, d, f), **f32)
        if glu:
            grads["dws_gate"] = torch.empty((S, f, d), **f32)
    scratch = torch.empty(max(moe.moe_expert_backward_scratch_size(cfg), 256), dtype=torch.uint8, device=dev)
    n_rs = moe.moe_route_backward_scratch_size(cfg)
    rscratch = torch.empty(n_rs, dtype=torch.uint8, device=dev) if n_rs else None
    gstruct = moe.make_expert_grads(grads)

    def comb():
        moe.moe_combine_backward(cfg, dy, y_perm, row_of, tw, dw, dy_perm, stream)

    def rout():
        moe.moe_route_backward(cfg, inp["x"], inp["w_router"], inp.get("logit_bias"), idx, tw, counts, dw, 1.0, 1.0,
                               dz, dwr, dx, rscratch, stream)

    def expert():
        moe.moe_expert_ffn_backward(cfg, weights, inp["x"], x_perm, offsets, row_of, dy, dy_perm, gstruct, dx,
                                    scratch, stream)

    def time_it(fn):
        for _ in range(2):
            fn()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        t0.record(stream)
        for _ in range(n):
            fn()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1) / n

    ms_c, ms_r, ms_e = time_it(comb), time_it(rout), time_it(expert)
    status = moe.moe_read_device_status(scratch)
    elt = 2 if wl.dtype == "bf16" else 4
    rows = int(offsets[E].item())
    comb_bytes = T * d * elt + rows * d * (4 + elt)          # dy in, kept rows of y_perm in, dy_perm out
    rout_flops = 3 * 2.0 * T * E * d                         # logits recomputed, dz^T x, dz W_r
    units = 7 if glu else 5                                  # recomputed pre-activations, dh, dW (x2-3), dx
    exp_flops = 2.0 * d * f * units * (rows + S * T)
    del ws, x_perm, y_perm, y_sh, dy_perm, dx, grads, scratch, rscratch
    return {"combine_backward_ms": round(ms_c, 4), "combine_backward_GB/s": round(comb_bytes / (ms_c * 1e-3) / 1e9, 1),
            "route_backward_ms": round(ms_r, 4),
            "route_backward_TFLOP/s": round(rout_flops / (ms_r * 1e-3) / 1e12, 2),
            "expert_backward_ms": round(ms_e, 4),
            "expert_backward_TFLOP/s": round(exp_flops / (ms_e * 1e-3) / 1e12, 1),
            "expert_backward_status": int(status),
            "note": "backward pass, each call timed alone, n=%d: combine backward on CUDA cores; router backward "
                    "%s; expert FFNs %s"
                    % (n, "on the tensor cores (dz as bf16 hi + lo)" if n_rs else "on fp32 CUDA cores",
                       "on the tensor cores (bf16 operands, fp32 accumulators and gradients)" if wl.dtype == "bf16"
                       else "on fp32 CUDA cores")}


def route_stats_of(moe, wl, cfg, inp, layer, drops, dev, stream):
    """Routing statistics of this workload (co-activation counts, imbalance, dropped share), from a
    standalone router call; timed alone, outside the layer's figures."""
    T = wl.T
    topk_idx = torch.empty((T, wl.k), dtype=torch.int32, device=dev)
    topk_w = torch.empty((T, wl.k), dtype=torch.float32, device=dev)
    r_counts = torch.empty(wl.E, dtype=torch.int32, device=dev)
    r_losses = torch.empty(2, dtype=torch.float32, device=dev)
    moe.moe_route(cfg, inp["x"], inp["w_router"], inp.get("logit_bias"), topk_idx, topk_w, r_counts, r_losses,
                  layer.ws, stream)
    coact = torch.empty((wl.E, wl.E), dtype=torch.int32, device=dev)
    rstats = torch.empty(2, dtype=torch.float32, device=dev)
    for _ in range(3):
        moe.moe_route_stats(cfg, topk_idx, None, coact, rstats, layer.ws, stream)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(10):
        moe.moe_route_stats(cfg, topk_idx, None, coact, rstats, layer.ws, stream)
    s1.record(stream)
    torch.cuda.synchronize(dev)
    cm = coact.double().cpu()
    diag = torch.diagonal(cm)
    score = torch.where(diag[:, None] > 0, cm / diag.clamp(min=1)[:, None], torch.zeros_like(cm))
    score.fill_diagonal_(0)
    return {"ms": round(s0.elapsed_time(s1) / 10, 5), "load_imbalance": round(float(rstats[0].item()), 4),
            "dropped_fraction": round(int(drops.item()) / (T * wl.k), 5),
            "max_coactivation_score": round(float(score.max().item()), 4)}


def e2e_of(moe, args, wl, cfg, inp, layer, y, counts, drops, dev, stream, ws_n):
    """End to end through the C ABI with host buffers (pinned), copies inside the timed region.
    As a serving loop would run them, the copies and the layer are pipelined over three streams
    (inputs in, compute, outputs out) with two device buffer sets: step i + 1's input copy and
    step i - 1's output copy overlap step i's layer.  Every step still copies its x in and its y
    and losses out inside the timed region."""
    NB = 2
    x_host = inp["x"].cpu().pin_memory()
    y_host = [torch.empty_like(x_host).pin_memory() for _ in range(NB)]
    l_host = [torch.empty(2, dtype=torch.float32).pin_memory() for _ in range(NB)]
    x_dev = [torch.empty_like(inp["x"]) for _ in range(NB)]
    y_dev = [torch.empty_like(inp["x"]) for _ in range(NB)]
    l_dev = [torch.empty(2, dtype=torch.float32, device=dev) for _ in range(NB)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(NB)]     # x_dev[b] holds this step's input
    ev_done = [torch.cuda.Event() for _ in range(NB)]   # the layer on buffer set b has finished
    ev_out = [torch.cuda.Event() for _ in range(NB)]    # y_dev[b] has been copied out

    def e2e_step(i):
        b = i % NB
        s_in.wait_event(ev_done[b])          # the layer that last read x_dev[b] is done
        with torch.cuda.stream(s_in):
            x_dev[b].copy_(x_host, non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])         # y_dev[b] has left for the host
        moe.moe_layer_forward(cfg, layer.weights, x_dev[b], y_dev[b], l_dev[b], counts, drops, layer.ws, stream)
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            y_host[b].copy_(y_dev[b], non_blocking=True)
            l_host[b].copy_(l_dev[b], non_blocking=True)
        ev_out[b].record(s_out)

    for i in range(max(2, args.warmup // 2)):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(args.steps):
        e2e_step(i)
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1)) / args.steps
    if not torch.equal(y_host[(args.steps - 1) % NB].to(dev), y):
        raise RuntimeError("end-to-end output differs from the device-resident run")
    st = moe.moe_read_device_status(layer.ws)
    if st != 0:
        raise RuntimeError(f"device status after the end-to-end run: {moe.moe_status_string(st)}")
    h2d = x_host.numel() * x_host.element_size()
    d2h = y_host[0].numel() * y_host[0].element_size() + 8
    return {"value": round(wl.T * ws_n / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "moe_layer_forward with pinned host x/y; copies in, layer and copies out pipelined "
                   "over three streams with two device buffer sets"}


def run_ours(args, wl, ws_n, rank, local):
    """The headline line: the workload it is quoted on, then (single GPU only) one sub-record per
    other workload, each with its own timing, stage times, roofline and CPU-oracle leg."""
    cpu = ws_n == 1 and not args.no_cpu_baseline
    head = measure(args, wl, ws_n, local, full=True, cpu_flops=3.0e11 if cpu else 0.0)
    res = {
        "metric": METRIC,
        "value": head["value"], "unit": "tokens/s",
        "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "eager": head["eager"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02^2) weights, random-init)",
        "config": arm_config(wl, ws_n),
    }
    for key in ("expert_tflops", "expert_frac_of_burst_peak", "expert_frac_of_sustained_peak", "stage_ms",
                "kept_rows", "drops", "roofline", "weight_stream", "route_stats", "backward", "e2e",
                "gpu_launches", "clocks", "stage_clocks", "cpu_baseline"):
        if key in head:
            res[key] = head[key]
    if ws_n == 1 and not args.no_per_config:
        res["per_config"] = {}
        for name in SUB_WORKLOADS:
            if name == wl.name:
                continue
            res["per_config"][name] = measure(args, WORKLOADS[name], ws_n, local, full=False,
                                              cpu_flops=4.0e10 if cpu else 0.0)
    return res


# ------------------------------------------------------------------------------ oracle (CPU)
def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [p.get("num_threads", 1) for p in threadpool_info() if p.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def oracle_step_fn(wl, tokens: int):
    """One oracle pass over the first ``tokens`` tokens of the workload (a bounded sample)."""
    from oracle import moe_oracle as O

    inp = make_inputs(wl.replace(T=tokens), "cpu")
    return lambda: O.moe_layer(inp, E=wl.E, k=wl.k, act=wl.act, n_shared=wl.n_shared, cf=wl.cf,
                               lb_coef=wl.lb_coef, z_coef=wl.z_coef)


def cpu_sample_tokens(wl, flops: float):
    """Tokens whose fp64 expert work is about ``flops``."""
    per_token = 2.0 * (wl.k + wl.n_shared) * (3 if wl.act == "swiglu" else 2) * wl.d * wl.dff
    return int(max(16, min(wl.T, flops / per_token)))


def run_reference(args, wl):
    n = cpu_sample_tokens(wl, 3.0e10)      # ~1-3 s per step on a few cores
    fn = oracle_step_fn(wl, n)
    per_step = []
    for i in range(args.warmup + max(1, args.steps)):
        t = time.perf_counter()
        fn()
        if i >= args.warmup:
            per_step.append(time.perf_counter() - t)
    ms = statistics.median(per_step) * 1e3
    value = n / (ms * 1e-3)
    cores = oracle_threads()
    sample = f"first {n} of {wl.T} tokens of {wl.name}, full layer in fp64 per step"
    return {
        "impl": "reference", "metric": METRIC,
        "value": round(value, 2), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": arm_config(wl, dist_env()[0]),
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def cpu_leg(wl, host_inp, n: int):
    """The oracle as it stands on the first ``n`` tokens of the workload's own tensors (already in
    host memory): the median of up to three passes (one when a pass takes over 3 s)."""
    from oracle import moe_oracle as O

    if getattr(wl, "weights8", "dtype") != "dtype":  # the oracle takes the dequantised weights
        deq = O.dequantize_rows_int8 if wl.weights8 == "int8" else O.dequantize_rows_e4m3
        host_inp = dict(host_inp)
        for wk, sk in (("w_up", "s_up"), ("w_gate", "s_gate"), ("w_down", "s_down"), ("ws_up", "ss_up"),
                       ("ws_gate", "ss_gate"), ("wb_up", "sb_up"), ("wb_gate", "sb_gate"), ("wb_down", "sb_down")):
            if host_inp.get(wk) is not None:
                host_inp[wk] = deq(host_inp[wk].numpy(), host_inp[sk].numpy())
        if host_inp.get("ws_down") is not None:  # one scale per row over the S matrices
            host_inp["ws_down"] = deq(host_inp["ws_down"].numpy(), host_inp["ss_down"].numpy()[None, :])
    times = []
    for _ in range(3):
        t = time.perf_counter()
        O.moe_layer(host_inp, E=wl.E, k=wl.k, act=wl.act, n_shared=wl.n_shared, cf=wl.cf, lb_coef=wl.lb_coef,
                    z_coef=wl.z_coef)
        times.append(time.perf_counter() - t)
        if times[-1] > 3.0:
            break
    sec = statistics.median(times)
    return {"value": round(n / sec, 2), "unit": "tokens/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"first {n} of {wl.T} tokens of {wl.name} (the benchmark's own tensors), full layer in "
                      f"fp64, median of {len(times)} pass(es) of {sec:.2f} s"}


# ------------------------------------------------------------------------------ distributed glue
_PG = False


def barrier():
    if _PG:
        torch.distributed.barrier()


def max_over_ranks(v: float) -> float:
    """The slowest rank's time (replicas are timed together; the job is as slow as its slowest)."""
    if not _PG:
        return v
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput of `world` replicas: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world / (ms_max * 1e-3)


def main():
    global _PG
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="only the headline workload")
    args = ap.parse_args()
    wl = WORKLOADS[args.workload]
    ws_n, rank, local = dist_env()

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, wl)), flush=True)
        return 0

    from mixture_experts_layer_89_b300 import build
    if rank == 0:
        build.build()
    if ws_n > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
        _PG = True
        barrier()
    res = run_ours(args, wl, ws_n, rank, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if _PG:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
