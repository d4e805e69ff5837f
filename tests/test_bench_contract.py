"""The benchmark's JSON line (CPU parts): the reference arm runs the oracle on the host and prints
the same metric, unit and workload config as the GPU arm; the L2 policy follows the weights."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import WORKLOADS  # noqa: E402


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0", "--workload", "tiny_fp32"], capture_output=True, text=True, timeout=300,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["config"] == bench.arm_config(WORKLOADS["tiny_fp32"], 1)
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_l2_policy_follows_the_weights():
    # weights under twice the L2 are flushed between steps; the large workloads stream more than L2
    assert bench.flushes_l2(WORKLOADS["tiny_fp32"])
    for name in ("flash_bf16", "finegrained_bf16", "decode_bf16", "skewed_bf16"):
        assert not bench.flushes_l2(WORKLOADS[name])
        assert bench.weight_bytes_of(WORKLOADS[name]) >= 2 * bench.L2_BYTES
    assert bench.weight_bytes_of(WORKLOADS["skewed_bf16"]) == 128 * 3 * 4096 * 6144 * 2


def test_expert_flops_counts_shared_experts():
    wl = WORKLOADS["finegrained_bf16"]
    up, down, sh_up, sh_down = bench.expert_flops(wl, wl.T * wl.k, wl.T)
    assert up == 2.0 * wl.T * wl.k * 2 * wl.d * wl.dff and down == up / 2
    assert sh_up == 2.0 * wl.T * wl.n_shared * 2 * wl.d * wl.dff and sh_down == sh_up / 2


def test_eight_bit_workloads_count_one_byte_per_weight():
    # 8-bit experts stream one byte per weight; the roofline adds their fp32 row scales
    for name in ("decode_int8_bf16", "skewed_int8_bf16"):
        wl8 = WORKLOADS[name]
        assert bench.weight_elt(wl8) == 1
        wl16 = wl8.replace(weights8="dtype")
        assert bench.weight_bytes_of(wl16) == 2 * bench.weight_bytes_of(wl8)
        assert "expert_weights" in bench.arm_config(wl8, 1) and "expert_weights" not in bench.arm_config(wl16, 1)
