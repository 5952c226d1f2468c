"""Host-side arithmetic of the benchmark line (no GPU): the roofline of a
kernel class counts the W_h bytes a recurrent step must read (state traffic
reported beside it, not in the denominator) against the copy bandwidth, and
the flops of the T*B-deep products against the burst bf16 peak; the roofline
of a whole step takes the slower of its flops and its recurrent weight reads."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from recurrent_neural_network_gb300 import synth  # noqa: E402

PK = dict(hbm_gbs=6788.3, bf16_tflops=1897.6, bf16_tflops_sustained=1716.1, sm_max_mhz=2070.0, source="measured")


def test_step_kernel_roofline_counts_only_the_recurrent_weights():
    wl = synth.WORKLOADS[3]  # 4-layer LSTM H=4096 B=256 T=50
    steps = 2
    n = 200 * steps
    us = 51.3
    r = bench.class_roofline("bwd_step", n, n * us * 1e-3, wl, steps, PK, True, True)
    wh = 4 * 4096 * 4096 * 2
    assert r["bytes_per_launch"] == wh
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(wh / (us * 1e-6) / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / PK["hbm_gbs"])
    assert r["frac"] == pytest.approx(0.3854, abs=1e-3)
    # the fp32 state traffic is reported beside the W_h bytes, not inside them
    assert r["state_bytes_per_launch"] > 0
    flops = 2.0 * 256 * 4 * 4096 * 4096
    assert r["flops_per_launch"] == pytest.approx(flops)
    assert r["tensor_frac"] == pytest.approx(flops / (us * 1e-6) / 1e12 / PK["bf16_tflops"])


def test_gemm_roofline_is_tensor_bound_against_the_burst_peak():
    wl = synth.WORKLOADS[3]
    steps = 3
    n = 4 * steps
    ms = 1.10
    r = bench.class_roofline("input_proj_gemm", n, n * ms, wl, steps, PK, True, True)
    flops = 2.0 * 50 * 256 * 4 * 4096 * 4096
    assert r["bound"] == "tensor" and r["peak"] == PK["bf16_tflops"]
    assert r["achieved"] == pytest.approx(flops / (ms * 1e-3) / 1e12)
    assert r["bytes_per_launch"] == 0


def test_workload_roofline_streaming_and_persistent():
    wl = synth.WORKLOADS[3]
    ms = 34.0
    r = bench.workload_roofline(wl, ms, PK, persistent=False)
    # 41.23 TF at the sustained peak (24 ms) binds over 400 W_h reads from HBM (7.9 ms)
    assert r["bound"] == "tensor"
    assert r["frac"] == pytest.approx(bench.step_flops(wl) / (PK["bf16_tflops_sustained"] * 1e12) / (ms * 1e-3))
    assert r["weight_bytes_per_step"] == 400 * 4 * 4096 * 4096 * 2
    p = synth.WORKLOADS[2]  # persistent B=4 H=1024 T=1000 inference
    r = bench.workload_roofline(p, 2.07, PK, persistent=True)
    assert r["bound"] == "smem"
    smem = 152 * 128 * 2070e6 / 1e9
    assert r["peak"] == pytest.approx(smem)
    roof_s = 1000 * 4 * 1024 * 1024 * 2 / (smem * 1e9)
    assert r["frac"] == pytest.approx(roof_s / 2.07e-3)
    f = synth.WORKLOADS[0]  # fp32: FFMA peak from the unit counts
    r = bench.workload_roofline(f, 0.5, PK, persistent=False)
    assert r["bound"] in ("alu", "hbm")
    assert r.get("tensor_frac", 0) >= 0


def test_workload_roofline_stacked_is_tensor_bound():
    """A stacked recurrence keeps its weights in tensor memory: the step is
    held to the sustained tensor peak."""
    wl = synth.WORKLOADS[1]  # 4-layer LSTM H=512 B=64 T=100 training
    r = bench.workload_roofline(wl, 1.4, PK, persistent=False, stacked=True)
    assert r["bound"] == "tensor" and r["peak"] == PK["bf16_tflops_sustained"]
    assert r["frac"] == pytest.approx(bench.step_flops(wl) / (PK["bf16_tflops_sustained"] * 1e12) / 1.4e-3)


def test_dp_aggregate_counts_every_rank():
    ms, tflops, w = bench.replica_aggregate(34.0, bench.step_flops(synth.WORKLOADS[3]))
    assert w == 1 and tflops == pytest.approx(41.23168604e12 / 34e-3 / 1e12, rel=1e-6)
