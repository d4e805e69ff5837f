"""GPU-vs-oracle parity of every step of the layer, through the C ABI (needs a B300).

Small and mid-sized cases span several tiles with ragged tails, capacity drops, shared experts,
exact ties, E = 1, k = E, E = 256 and a single token; the full workloads run in the launch
configuration the benchmark times.  Inputs are drawn once by ``synth.make_inputs``; the same
tensors go to the library and (as host copies) to the oracle.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_89_b300 import moe
from oracle import moe_oracle as O
from synth import WORKLOADS, Workload, make_inputs

from parity_utils import (check_losses, check_output, check_topk_weights, dispatch_is_valid, oracle, routing_report,
                          run_layer, run_steps, to_np)

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_fp32": WORKLOADS["tiny_fp32"],
    "fp32_gelu_bias_ragged": Workload("fp32_gelu_bias_ragged", T=333, d=96, E=6, k=3, dff=160, act="gelu",
                                      dtype="f32", bias=True, bias_std=0.02, seed=11, wseed=11),
    "fp32_swiglu_shared_cap": Workload("fp32_swiglu_shared_cap", T=257, d=64, E=8, k=2, dff=128, act="swiglu",
                                       dtype="f32", n_shared=2, cf=1.0, seed=12, wseed=12),
    "fp32_E256_k8": Workload("fp32_E256_k8", T=100, d=40, E=256, k=8, dff=24, act="gelu", dtype="f32",
                             seed=20, wseed=20),
    "bf16_gelu_bias_ragged": Workload("bf16_gelu_bias_ragged", T=1000, d=256, E=8, k=2, dff=512, act="gelu",
                                      dtype="bf16", bias=True, bias_std=0.02, cf=1.1, seed=13, wseed=13),
    "bf16_swiglu_shared": Workload("bf16_swiglu_shared", T=700, d=512, E=16, k=4, dff=256, act="swiglu",
                                   dtype="bf16", n_shared=2, cf=1.25, seed=14, wseed=14),
    "bf16_k_eq_E": Workload("bf16_k_eq_E", T=130, d=128, E=4, k=4, dff=128, act="swiglu", dtype="bf16",
                            seed=15, wseed=15),
    "bf16_E1": Workload("bf16_E1", T=200, d=64, E=1, k=1, dff=64, act="gelu", dtype="bf16", seed=16, wseed=16),
    "bf16_collapse_cap": Workload("bf16_collapse_cap", T=300, d=128, E=8, k=2, dff=128, act="swiglu",
                                  dtype="bf16", cf=1.0, logit_bias0=50.0, seed=17, wseed=17),
    "bf16_one_token": Workload("bf16_one_token", T=1, d=128, E=8, k=2, dff=128, act="swiglu", dtype="bf16",
                               n_shared=1, seed=18, wseed=18),
    "bf16_E256_k8": Workload("bf16_E256_k8", T=512, d=128, E=256, k=8, dff=64, act="swiglu", dtype="bf16",
                             seed=19, wseed=19),
    "bf16_gelu_shared3": Workload("bf16_gelu_shared3", T=260, d=192, E=5, k=2, dff=256, act="gelu",
                                  dtype="bf16", n_shared=3, seed=21, wseed=21),
    # capacity 1: every expert keeps only its first assignment in token order
    "bf16_cap1": Workload("bf16_cap1", T=300, d=128, E=8, k=2, dff=128, act="swiglu", dtype="bf16",
                          n_shared=1, cf=0.01, seed=23, wseed=23),
    # enough rows per expert for the paired (2-SM) projections, with non-zero biases and drops
    "bf16_gelu_bias_pair": Workload("bf16_gelu_bias_pair", T=2100, d=256, E=4, k=2, dff=512, act="gelu",
                                    dtype="bf16", bias=True, bias_std=0.02, cf=1.05, seed=22, wseed=22),
    # router temperature (a routing variant): softmax, weights and losses of z / tau
    "bf16_swiglu_temp2": Workload("bf16_swiglu_temp2", T=700, d=512, E=16, k=4, dff=256, act="swiglu",
                                  dtype="bf16", n_shared=2, cf=1.25, seed=24, wseed=24, temperature=2.0),
    "fp32_gelu_temp_half": Workload("fp32_gelu_temp_half", T=150, d=64, E=8, k=2, dff=128, act="gelu",
                                    dtype="f32", bias=True, seed=25, wseed=25, temperature=0.5),
}


def _to(inp, dev):
    return {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}


def _shared_ref(wl, inp_cpu, tokens):
    if not wl.n_shared:
        return None
    x = O._f64(inp_cpu["x"])[tokens]
    ys = np.zeros((len(tokens), wl.d))
    for s in range(wl.n_shared):
        g = None if inp_cpu.get("ws_gate") is None else inp_cpu["ws_gate"][s]
        ys += O.expert_ffn(x, wl.act, inp_cpu["ws_up"][s], inp_cpu["ws_down"][s], g)
    return ys


def check_all_steps(wl, inp_cpu, inp_gpu, tokens=None):
    got = run_steps(wl, inp_gpu)
    assert got["status"] == moe.MOE_OK, moe.moe_status_string(got["status"])
    ref = oracle(wl, inp_cpu, tokens=tokens)
    T = inp_cpu["x"].shape[0]
    gidx = got["topk_idx"].cpu().numpy().astype(np.int64)
    gw = got["topk_w"].cpu().numpy().astype(np.float64)
    n_b, n_o = routing_report(gidx, ref, wl.k)
    bexempt = ref["gap"] < 1e-5
    check_topk_weights(gidx, gw, ref, bexempt)
    check_losses(got["losses"], ref["lb"], ref["zl"])
    counts = got["counts"].cpu().numpy()
    offsets = got["offsets"].cpu().numpy()
    kept = got["kept"].cpu().numpy()
    row_of = got["row_of"].cpu().numpy()
    tok_of = got["tok_of"].cpu().numpy()
    A = int(offsets[-1])
    assert A <= got["amax"]
    if n_b == 0:
        assert np.array_equal(counts, ref["counts"])
        assert np.array_equal(kept, ref["kept_counts"])
        assert np.array_equal(offsets, ref["offsets"])
        assert np.array_equal(row_of, ref["row_of"])
        assert np.array_equal(tok_of[:A], ref["tok_of"])
    dispatch_is_valid(gidx, wl.E, got["cap"], counts, offsets, kept, row_of, tok_of)
    # dispatch copies rows bit for bit
    if A:
        assert torch.equal(got["x_perm"][:A], inp_gpu["x"][got["tok_of"][:A].long()])
    # tokens whose routing (selected set and kept flags) equals the oracle's
    same = np.array([sorted(gidx[t]) == sorted(ref["idx"][t]) and
                     sorted(gidx[t][row_of[t] >= 0]) == sorted(ref["idx"][t][ref["row_of"][t] >= 0])
                     for t in range(T)], dtype=bool)
    toks = ref["tokens"]
    if n_b == 0:
        assert same.all()
        # expert outputs per sorted row (oracle rows of the sampled tokens)
        tokset = set(toks.tolist())
        rows = [r for r in range(A) if int(ref["tok_of"][r]) in tokset]
        if rows:
            check_output(to_np(got["y_perm"][rows]), ref["y_perm"][rows], wl.dtype, "y_perm")
    ys_ref = _shared_ref(wl, inp_cpu, toks)
    if ys_ref is not None:
        check_output(to_np(got["y_shared"][torch.as_tensor(toks, device=inp_gpu["x"].device)]), ys_ref, wl.dtype,
                     "y_shared")
    sel = same[toks]
    y = to_np(got["y"])[toks]
    check_output(y[sel], ref["y"][sel], wl.dtype, "y")
    return got, ref, n_b, n_o


@pytest.mark.parametrize("case", list(CASES))
def test_steps_match_oracle(case):
    wl = CASES[case]
    inp_cpu = make_inputs(wl, "cpu")
    inp_gpu = _to(inp_cpu, "cuda")
    got, ref, n_b, n_o = check_all_steps(wl, inp_cpu, inp_gpu)
    print(f"{case}: boundary-exempt tokens {n_b}, order-exempt tokens {n_o}, drops {ref['drops']}")
    # the whole-layer entry point runs the same kernels in the same order: identical results
    lay = run_layer(wl, inp_gpu)
    assert lay["status"] == moe.MOE_OK
    assert torch.equal(lay["y"], got["y"])
    assert torch.equal(lay["losses"], got["losses"])
    assert torch.equal(lay["counts"], got["counts"])
    assert int(lay["drops"].item()) == wl.T * wl.k - int(got["offsets"][-1].item())


def test_all_ties_pick_lowest_indices():
    wl = CASES["bf16_swiglu_shared"].replace(T=64)
    inp_cpu = make_inputs(wl, "cpu")
    inp_cpu["x"][::2] = 0          # even tokens: every logit is exactly 0
    got = run_steps(wl, _to(inp_cpu, "cuda"))
    idx = got["topk_idx"].cpu().numpy()
    w = got["topk_w"].cpu().numpy()
    for t in range(0, 64, 2):
        assert idx[t].tolist() == list(range(wl.k))
        assert np.allclose(w[t], 1.0 / wl.k, atol=1e-7)
    check_all_steps(wl, inp_cpu, _to(inp_cpu, "cuda"))


def test_small_router_near_ties_decided_exactly():
    """Decode-sized calls route on fp32 logits with an error bound and recompute a token's logits
    with compensated sums when its leading logits lie within the bounds.  Experts 0 and 1 differ by
    one bf16 step in one weight and carry the same large logit bias, so every token's top two are
    {0, 1} with a gap of |x_tj| * 2^-13 -- mostly above the 1e-5 exemption yet below the fp32
    bound (~2e-4 here): the order must be the exact one."""
    wl = Workload("bf16_near_ties", T=48, d=2048, E=16, k=2, dff=128, act="swiglu", dtype="bf16", seed=31, wseed=31)
    inp_cpu = make_inputs(wl, "cpu")
    w = inp_cpu["w_router"].float()
    j = 5
    w[1] = w[0]
    w[0, j] = 0.02
    w[1, j] = 0.02 + 2.0 ** -13          # one bf16 step above 0.02 (spacing 2^-13 in [2^-6, 2^-5))
    inp_cpu["w_router"] = w.to(torch.bfloat16)
    assert float(inp_cpu["w_router"][1, j]) - float(inp_cpu["w_router"][0, j]) == 2.0 ** -13
    lb = torch.zeros(wl.E)
    lb[:2] = 5.0
    inp_cpu["logit_bias"] = lb
    ref = oracle(wl, inp_cpu)
    gap = np.abs(O._f64(inp_cpu["x"])[:, j]) * 2.0 ** -13
    assert (gap > 1e-5).sum() >= 40 and ((gap > 1e-5) & (gap < 1e-4)).sum() >= 25  # most below the fp32 bound
    assert all(sorted(ref["idx"][t].tolist()) == [0, 1] for t in range(wl.T))
    got = run_steps(wl, _to(inp_cpu, "cuda"))
    assert got["status"] == moe.MOE_OK
    idx = got["topk_idx"].cpu().numpy()
    assert all(sorted(idx[t].tolist()) == [0, 1] for t in range(wl.T))
    decided = gap > 1e-5               # the exemption applies to the rest: either order is acceptable
    bad = np.nonzero((idx != ref["idx"]).any(axis=1) & decided)[0]
    assert bad.size == 0, [(int(t), idx[t].tolist(), ref["idx"][t].tolist(), float(gap[t])) for t in bad]
    check_topk_weights(idx, got["topk_w"].cpu().numpy().astype(np.float64), ref, np.zeros(wl.T, bool))
    check_losses(got["losses"], ref["lb"], ref["zl"])


def test_empty_batch():
    wl = CASES["bf16_swiglu_shared"].replace(T=0)
    inp_gpu = _to(make_inputs(wl, "cpu"), "cuda")
    got = run_steps(wl, inp_gpu, T=0)
    assert got["status"] == moe.MOE_OK
    assert got["counts"].sum().item() == 0 and got["offsets"].abs().sum().item() == 0
    assert got["losses"].abs().sum().item() == 0
    lay = run_layer(wl, inp_gpu)
    assert lay["status"] == moe.MOE_OK and lay["y"].numel() == 0 and int(lay["drops"].item()) == 0


def test_nonfinite_input_is_reported():
    wl = CASES["bf16_k_eq_E"]
    inp = _to(make_inputs(wl, "cpu"), "cuda")
    inp["x"][3, 5] = float("nan")
    got = run_steps(wl, inp)
    assert got["status"] == moe.MOE_ERR_DEVICE_STATUS
    idx = got["topk_idx"].cpu().numpy()
    assert ((idx >= 0) & (idx < wl.E)).all()   # indices stay valid, nothing runs out of bounds


def test_bad_counts_are_reported():
    wl = CASES["bf16_gelu_bias_ragged"]
    inp = _to(make_inputs(wl, "cpu"), "cuda")
    cfg = moe.config_from_workload(wl)
    got = run_steps(wl, inp)
    ws = moe.alloc_workspace(cfg)
    bad = got["counts"].clone()
    bad[0] += 1
    amax = got["amax"]
    z = lambda n: torch.zeros(n, dtype=torch.int32, device="cuda")
    moe.moe_permute(cfg, inp["x"], got["topk_idx"], bad, z(wl.E + 1), z(wl.E), z(wl.T * wl.k), z(amax),
                    torch.zeros_like(got["x_perm"]), ws)
    assert moe.moe_read_device_status(ws) == moe.MOE_ERR_DEVICE_STATUS
    assert moe.moe_read_device_status(ws) == moe.MOE_OK   # reading clears it


def test_forced_router_timeout_is_reported_and_recovers():
    """A bounded device wait made to run out.  The router's waits are shortened to 1 ns through the
    workspace, so its first wait for a TMA copy gives up: the CTA lets its copies and MMAs in flight
    finish, records MOE_ERR_TIMEOUT in the status word and returns, and the GPU stays usable.  With
    the default limit restored, the same workspace routes exactly as before."""
    wl = CASES["bf16_swiglu_shared"]
    inp = _to(make_inputs(wl, "cpu"), "cuda")
    cfg = moe.config_from_workload(wl)
    ws = moe.alloc_workspace(cfg)

    def route():
        T, E, k = cfg.T, cfg.E, cfg.k
        out = dict(idx=torch.full((T, k), -7, dtype=torch.int32, device="cuda"),
                   w=torch.full((T, k), -1.0, dtype=torch.float32, device="cuda"),
                   counts=torch.full((E,), -7, dtype=torch.int32, device="cuda"),
                   losses=torch.full((2,), -1.0, dtype=torch.float32, device="cuda"))
        moe.moe_route(cfg, inp["x"], inp["w_router"], inp.get("logit_bias"), out["idx"], out["w"], out["counts"],
                      out["losses"], ws)
        return out

    ref = route()
    assert moe.moe_read_device_status(ws) == moe.MOE_OK
    moe.moe_set_wait_limit(ws, 1)
    route()
    assert moe.moe_read_device_status(ws) == moe.MOE_ERR_TIMEOUT
    moe.moe_set_wait_limit(ws, 0)
    got = route()
    assert moe.moe_read_device_status(ws) == moe.MOE_OK
    for name in ref:
        assert torch.equal(ref[name], got[name]), name


def test_repeat_calls_are_deterministic():
    wl = CASES["bf16_swiglu_shared"]
    inp = _to(make_inputs(wl, "cpu"), "cuda")
    a = run_layer(wl, inp)
    b = run_layer(wl, inp)
    assert torch.equal(a["y"], b["y"]) and torch.equal(a["losses"], b["losses"])


def test_graph_replay_matches_eager():
    """The layer captured in a CUDA graph (small shared experts fork onto a second stream and join
    back before the combine) reproduces the eager result bit for bit, also after new inputs are
    copied into the captured buffer."""
    wl = CASES["bf16_swiglu_shared"]
    inp = _to(make_inputs(wl, "cpu"), "cuda")
    layer = moe.MoELayer(moe.config_from_workload(wl), inp)
    x = inp["x"].clone()
    ref1 = layer.forward(x)
    ref2 = layer.forward(x.flip(0).contiguous())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = layer.forward(x, stream=torch.cuda.current_stream())
    for ref, src in ((ref1, inp["x"]), (ref2, inp["x"].flip(0))):
        x.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        assert moe.moe_read_device_status(layer.ws) == moe.MOE_OK
        for a, b in zip(out, ref):
            assert torch.equal(a, b)


def _check_route_stats(wl, inp_gpu, got):
    cfg = moe.config_from_workload(wl, inp_gpu["x"].shape[0])
    ws = moe.alloc_workspace(cfg)
    coact = torch.full((wl.E, wl.E), -7, dtype=torch.int32, device="cuda")
    stats = torch.full((2,), -1.0, dtype=torch.float32, device="cuda")
    moe.moe_route_stats(cfg, got["topk_idx"], got["offsets"], coact, stats, ws)
    assert moe.moe_read_device_status(ws) == moe.MOE_OK
    idx = got["topk_idx"].cpu().numpy()
    assert np.array_equal(coact.cpu().numpy(), O.coactivation(idx, wl.E))      # integer counts: exact
    imb, drop = O.routing_stats(idx, wl.E, wl.k, got["offsets"].cpu().numpy())
    np.testing.assert_allclose(stats.cpu().numpy(), [imb, drop], rtol=1e-6)


@pytest.mark.parametrize("case", ["bf16_swiglu_shared", "bf16_collapse_cap", "bf16_E256_k8", "fp32_E256_k8",
                                  "bf16_one_token"])
def test_route_stats_match_oracle(case):
    """Co-activation counts (shared-memory path for E <= 128, global atomics above), load
    imbalance and dropped fraction, from the library's own top-k indices and offsets."""
    wl = CASES[case]
    inp = _to(make_inputs(wl, "cpu"), "cuda")
    got = run_steps(wl, inp)
    assert got["status"] == moe.MOE_OK
    _check_route_stats(wl, inp, got)


def test_route_stats_empty_batch():
    wl = CASES["bf16_swiglu_shared"].replace(T=0)
    cfg = moe.config_from_workload(wl)
    ws = moe.alloc_workspace(cfg)
    coact = torch.full((wl.E, wl.E), -7, dtype=torch.int32, device="cuda")
    stats = torch.full((2,), -1.0, dtype=torch.float32, device="cuda")
    moe.moe_route_stats(cfg, None, None, coact, stats, ws)
    assert coact.abs().sum().item() == 0 and stats.abs().sum().item() == 0


# ------------------------------------------------------------------------------ full workloads
def _full(name, n_sample, seed=0):
    wl = WORKLOADS[name]
    inp_gpu = make_inputs(wl, "cuda")
    torch.cuda.synchronize()
    rng = np.random.default_rng(seed)
    toks = None if n_sample is None else np.sort(rng.choice(wl.T, size=min(n_sample, wl.T), replace=False))
    got, ref, n_b, n_o = check_all_steps(wl, inp_gpu, inp_gpu, tokens=toks)
    print(f"{name}: boundary-exempt {n_b}, order-exempt {n_o}, drops {ref['drops']}, cap {ref['cap']}, "
          f"expert-0 share {ref['counts'][0] / wl.T:.3f}")
    return got, ref


def test_full_flash_bf16():
    _full("flash_bf16", None)


def test_route_stats_full_finegrained():
    wl = WORKLOADS["finegrained_bf16"]
    inp = make_inputs(wl, "cuda")
    got = run_steps(wl, inp)
    assert got["status"] == moe.MOE_OK
    _check_route_stats(wl, inp, got)


def test_full_finegrained_bf16():
    _full("finegrained_bf16", None)


def test_full_decode_bf16():
    _full("decode_bf16", None)


@pytest.mark.slow
def test_full_skewed_bf16():
    # 19.3 GB of weights: routing, dispatch and losses on every token, the layer output (and the
    # expert rows feeding it) on a seeded sample of 1024 tokens
    _full("skewed_bf16", 1024)


@pytest.mark.slow
def test_full_skewed_cf1_bf16():
    got, ref = _full("skewed_cf1_bf16", 1024, seed=1)
    assert ref["drops"] > 0


# ------------------------------------------------------------------------------ routing diagnostics
def _check_diagnostics(wl, inp_gpu, inp_cpu=None):
    inp_cpu = inp_gpu if inp_cpu is None else inp_cpu
    T = inp_gpu["x"].shape[0]
    cfg = moe.config_from_workload(wl, T)
    ws = moe.alloc_workspace(cfg)
    diag = torch.full((4,), -1.0, dtype=torch.float32, device="cuda")
    ent = torch.full((max(T, 1),), -1.0, dtype=torch.float32, device="cuda")
    moe.moe_route_diagnostics(cfg, inp_gpu["x"], inp_gpu["w_router"], inp_gpu.get("logit_bias"), diag, ent, ws)
    assert moe.moe_read_device_status(ws) == moe.MOE_OK
    z = O.temper(O.router_logits(inp_cpu["x"], inp_cpu["w_router"], inp_cpu.get("logit_bias")), wl.temperature)
    P, lse = O.softmax_lse(z)
    h_tok = lse - np.sum(P * z, axis=1) if T else np.zeros(0)
    got = diag.cpu().numpy().astype(np.float64)
    if T == 0:
        assert np.all(got == 0)
        return
    idx = O.topk_select(z, wl.k)
    counts = np.bincount(idx.ravel(), minlength=wl.E)
    ref = [float(np.mean(h_tok)), O.lb_loss_squared_mean_form(P, wl.lb_coef),
           O.lb_loss_kl_frequency_form(P, counts, wl.lb_coef), O.aux_losses(P, lse, counts, wl.k, wl.lb_coef, 0.0)[0]]
    np.testing.assert_allclose(ent[:T].cpu().numpy(), h_tok, rtol=1e-4, atol=2e-5)
    # near-tie tokens (oracle gap < 1e-5) may fall on either side of the top-k boundary: each moves
    # one count, 1 / (T k) of f
    n_exempt = int((O.topk_gap(z, wl.k) < 1e-5).sum())
    np.testing.assert_allclose(got[:2], ref[:2], rtol=1e-4, atol=1e-7)
    tol = 1e-4 + 4.0 * n_exempt / (T * wl.k)
    np.testing.assert_allclose(got[2:], ref[2:], rtol=tol, atol=1e-7)
    print(f"  diagnostics {wl.name}: {got.tolist()} vs {ref}; near ties {n_exempt}")


@pytest.mark.parametrize("case", ["bf16_swiglu_shared", "bf16_E256_k8", "fp32_E256_k8", "bf16_collapse_cap",
                                  "bf16_swiglu_temp2", "fp32_gelu_temp_half", "bf16_one_token", "tiny_fp32"])
def test_route_diagnostics_match_oracle(case):
    """Router entropy (per token and mean) and the three balance-loss forms, against the oracle's
    router_entropy, lb_loss_squared_mean_form, lb_loss_kl_frequency_form and aux_losses."""
    wl = CASES[case]
    inp_cpu = make_inputs(wl, "cpu")
    _check_diagnostics(wl, _to(inp_cpu, "cuda"), inp_cpu)


def test_route_diagnostics_empty_batch():
    wl = CASES["bf16_swiglu_shared"].replace(T=0)
    _check_diagnostics(wl, _to(make_inputs(wl, "cpu"), "cuda"))


def test_route_diagnostics_full_finegrained():
    wl = WORKLOADS["finegrained_bf16"]
    _check_diagnostics(wl, make_inputs(wl, "cuda"))


# ------------------------------------------------------------------------------ backup expert
BACKUP_CASES = {
    "bf16_swiglu_backup": Workload("bf16_swiglu_backup", T=700, d=512, E=16, k=4, dff=256, act="swiglu",
                                   dtype="bf16", n_shared=2, cf=0.6, seed=26, wseed=26, backup=True),
    "bf16_gelu_bias_backup": Workload("bf16_gelu_bias_backup", T=1000, d=256, E=8, k=2, dff=512, act="gelu",
                                      dtype="bf16", bias=True, bias_std=0.02, cf=0.7, seed=27, wseed=27,
                                      backup=True),
    "bf16_collapse_backup": Workload("bf16_collapse_backup", T=300, d=128, E=8, k=2, dff=128, act="swiglu",
                                     dtype="bf16", cf=1.0, logit_bias0=50.0, seed=28, wseed=28, backup=True),
    "fp32_gelu_backup": Workload("fp32_gelu_backup", T=333, d=96, E=6, k=3, dff=160, act="gelu", dtype="f32",
                                 bias=True, bias_std=0.02, cf=0.5, seed=29, wseed=29, backup=True),
    "bf16_decode_backup": Workload("bf16_decode_backup", T=32, d=256, E=8, k=2, dff=256, act="swiglu",
                                   dtype="bf16", n_shared=1, cf=0.5, seed=30, wseed=30, backup=True),
}


@pytest.mark.parametrize("case", list(BACKUP_CASES))
def test_backup_expert_matches_oracle(case):
    """Assignments over capacity go, with their routing weight, to one extra expert: the dispatch
    places them after the kept rows in (token, slot) order, the projections run the backup expert on
    them in the same launches, and the combine adds them -- against the oracle's
    moe_layer_backup_expert on the same tensors."""
    wl = BACKUP_CASES[case]
    inp_cpu = make_inputs(wl, "cpu")
    inp_gpu = _to(inp_cpu, "cuda")
    backup = {n: inp_cpu[m] for n, m in (("w_up", "wb_up"), ("w_gate", "wb_gate"), ("w_down", "wb_down"),
                                         ("b_up", "bb_up"), ("b_down", "bb_down"))}
    ref = O.moe_layer_backup_expert(inp_cpu, backup, E=wl.E, k=wl.k, act=wl.act, n_shared=wl.n_shared, cf=wl.cf,
                                    lb_coef=wl.lb_coef, z_coef=wl.z_coef)
    assert ref["backup_rows"] > 0 and (ref["gap"] >= 1e-5).all()
    got = run_steps(wl, inp_gpu)
    assert got["status"] == moe.MOE_OK, moe.moe_status_string(got["status"])
    T, k, E = wl.T, wl.k, wl.E
    A = int(ref["offsets"][E])
    assert np.array_equal(got["offsets"].cpu().numpy(), ref["offsets"])
    # kept rows as without the backup; the dropped slots, in (token, slot) order, at A, A + 1, ...
    row_of = got["row_of"].cpu().numpy()
    exp_rows = ref["row_of"].copy()
    dropped = exp_rows < 0
    exp_rows[dropped] = A + np.arange(int(dropped.sum()))
    assert np.array_equal(row_of, exp_rows)
    tok_of = got["tok_of"].cpu().numpy()
    assert np.array_equal(tok_of[A:T * k], np.nonzero(dropped)[0])
    assert torch.equal(got["x_perm"][:T * k], inp_gpu["x"][got["tok_of"][:T * k].long()])
    check_losses(got["losses"], ref["lb"], ref["zl"])
    check_output(to_np(got["y"]), ref["y"], wl.dtype, "y")
    lay = run_layer(wl, inp_gpu)
    assert lay["status"] == moe.MOE_OK
    assert torch.equal(lay["y"], got["y"])
    assert int(lay["drops"].item()) == ref["drops"]
