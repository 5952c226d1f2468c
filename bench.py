"""Benchmark of the stacked-RNN hot path on GB300.

One step = one full pass of the path over one batch of seeded synthetic
input: for a training workload the forward pass (input projection, fused
recurrent steps, layer wavefront), the backward pass through time (fused
reverse steps, data-gradient products) and the weight-gradient products; for
an inference workload the forward pass.  Default workload: the 4-layer
H=4096 B=256 T=50 bf16 LSTM training step.

    python bench.py [--gpus N --steps K --warmup W] [--config IDX] [--impl reference]

Prints one JSON line (rank 0).  Metric: algorithmic GEMM TFLOP/s of the step
(2*M*N*K over the input, recurrent, data-gradient and weight-gradient
products), with timesteps/s beside it.  With N > 1 (torchrun, one rank per
GPU) the step is data-parallel: the global batch holds N shards of the
workload's batch, every rank runs its shard and the weight gradients are
summed over the ranks with one NCCL all-reduce per step inside the timed
region (weak scaling: per-GPU work is fixed).  Inference workloads have no
exchange step and run one shard per rank.

Besides the headline workload the line carries measured sub-results of the
other benchmark workloads ("workloads"), each with its roofline fraction.
Moderate batches (9..64 sequences: the 4-layer H=512 B=64 LSTM and the
8-layer H=1024 B=32 GRU) run the persistent stacked recurrences, whose plan
string the sub-result carries.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "LSTM fwd+bwd TFLOPS & timesteps/s on 1 GB300; % of bf16 tensor/SMEM roofline"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d.get("hbm_gbs", 6800.0), bf16_tflops=d.get("bf16_tflops", 1900.0),
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", 1700.0), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        # raw samples go to a scratch file; the JSON line carries their summary
        self.path = os.path.join(tempfile.gettempdir(), f"clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            try:
                pw.append(float(parts[3]))
            except ValueError:
                pass
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "power_w": statistics.median(pw) if pw else None, "reasons": sorted(reasons)}


def replica_aggregate(ms_local, flops_per_step, dist=None, device="cpu"):
    """Whole-job throughput of N independent replicas: every rank processed
    one workload per step; the step time is the maximum over ranks.  Returns
    (max ms per step, aggregate TFLOP/s, world size)."""
    world = 1
    ms = float(ms_local)
    if dist is not None and dist.is_initialized():
        world = dist.get_world_size()
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * flops_per_step / (ms * 1e-3) / 1e12, world


def step_flops(wl):
    f = wl.gemm_flops()
    return f["fwd"] + (f["bwd_data"] + f["bwd_weights"] if wl.training else 0.0)


def class_flops(wl):
    """Algorithmic flops per step of each kernel class (for the roofline of the dominant one)."""
    G, H, T, B, L = wl.G, wl.hidden, wl.T, wl.B, wl.layers
    inp = sum(2.0 * T * B * G * H * wl.in_size(l) for l in range(L))
    rec = 2.0 * T * B * G * H * H * L
    out = {"input_proj_gemm": inp, "fwd_step": rec}
    if wl.training:
        out.update({"bwd_step": rec, "dx_gemm": inp, "dw_gemm": inp + rec})
    return out


def class_bytes(wl, transposed, fused_point=False):
    """Algorithmic HBM bytes per step of the recurrent-step classes: every
    timestep reads W_h once plus the state it updates (bf16 storage, f32 gates,
    cell state and gate pre-activations).  With transposed steps the BPTT
    product only writes dh and a pointwise kernel (bwd_point) does the rest."""
    G, H, T, B, L = wl.G, wl.hidden, wl.T, wl.B, wl.layers
    e = 2 if wl.mode == 1 else 4
    wh = G * H * H * e
    # forward: h_{t-1} + P (read) ; gates (write) ; c_{t-1}/c_t ; h_t, y
    fwd = wh + B * H * e + B * G * H * 4 * 2 + B * H * 4 * 2 + B * H * e * 2
    out = {"fwd_step": fwd * T * L}
    if not wl.training:
        return out
    if transposed:
        # pointwise: dy, gates, c_s, c_{s-1}, carry (read) ; dG_s, carry (write)
        point = B * H * 4 + B * G * H * 4 + B * H * 4 * 2 + B * H * 4 * 2 + B * G * H * e
        if fused_point:
            # product with the pointwise step in its epilogue: W_h + dG_{s+1} + pointwise inputs and outputs
            out["bwd_step"] = (wh + B * G * H * e + point) * T * L
            out["bwd_point"] = (B * H * 4 + point) * L  # only the last timestep runs it alone
        else:
            # product: W_h + dG_{s+1} (read) ; dh (write).  pointwise: dh (read) + the rest
            out["bwd_step"] = (wh + B * G * H * e + B * H * 4) * T * L
            out["bwd_point"] = (B * H * 4 + point) * T * L
    else:
        # fused: dG_{t+1} + gates + c_t, c_{t-1} + dy + carry (read) ; dG_t + carry (write)
        out["bwd_step"] = (wh + B * G * H * e + B * G * H * 4 + B * H * 4 * 2 + B * H * 4 * 2 + B * G * H * e
                           + B * H * 4) * T * L
    return out


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture of the same kernel build on `bench.py --ncu-steps` (one layer,
# T=2, the same per-step shape; transposed steps, BPTT pointwise fused into the
# product): the first launch of each class.
NCU_TRAFFIC = {("lstm_bf16_L4_T50_B256_H4096", "bwd_step"): 177.24e6,
               ("lstm_bf16_L4_T50_B256_H4096", "fwd_step"): 162.46e6}


def oracle_sample(wl, B1, T1):
    """The double-precision oracle on batch columns 0..B1-1 and timesteps
    0..T1-1 of the workload (all layers); returns (cpu_baseline dict, seconds)."""
    import oracle
    from recurrent_neural_network_gb300 import runner
    sw = wl.replace(B=B1, T=T1)
    hi = runner.HostInputs(sw)
    t0 = time.perf_counter()
    if wl.training:
        oracle.bwd(sw.cell, sw.layers, sw.T, sw.B, sw.input, sw.hidden, hi.x, hi.w, hi.dy, h0=hi.h0, c0=hi.c0,
                   D=sw.directions)
    else:
        oracle.fwd(sw.cell, sw.layers, sw.T, sw.B, sw.input, sw.hidden, hi.x, hi.w, h0=hi.h0, c0=hi.c0,
                   D=sw.directions)
    dt = time.perf_counter() - t0
    fl = step_flops(sw)
    return dict(value=fl / dt / 1e12, unit="TFLOP/s", cores=oracle.threads(), kind="oracle",
                sample=f"B={B1} of {wl.B} columns, T={T1} of {wl.T} steps, all {wl.layers} layers "
                       f"({'fwd+BPTT+dW' if wl.training else 'fwd'}), {dt:.2f} s"), dt


def oracle_sample_shape(wl, budget_s):
    """(B1, T1) for an oracle run of about budget_s seconds: timed on a small
    sample first, then grown along the timesteps and then the batch."""
    B0 = min(wl.B, 2)
    T0 = min(wl.T, 4 if wl.hidden >= 2048 else 16)
    _, dt0 = oracle_sample(wl, B0, T0)
    f = budget_s / max(dt0, 1e-3)
    T1 = min(wl.T, max(T0, int(T0 * f)))
    B1 = min(wl.B, max(B0, int(B0 * f * T0 / T1)))
    return B1, T1


def time_oracle_sample(wl, budget_s=12.0):
    """cpu_baseline: the oracle as it stands on about budget_s seconds of the workload."""
    B1, T1 = oracle_sample_shape(wl, budget_s)
    return oracle_sample(wl, B1, T1)


def run_reference(args, wl, rank):
    """--impl reference: the oracle timed on host cores, per step one bounded
    sample sized so that warm-up and timed steps together take a few minutes."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    per_step = min(20.0, max(1.5, 150.0 / max(1, args.warmup + args.steps)))
    B1, T1 = oracle_sample_shape(wl, per_step)
    times = []
    res = None
    for i in range(args.warmup + args.steps):
        res, dt = oracle_sample(wl, B1, T1)
        if i >= args.warmup:
            times.append(dt)
    ms = 1e3 * statistics.mean(times)
    line = {"impl": "reference", "metric": METRIC, "value": res["value"], "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, "sample": res["sample"]},
            "cpu_baseline": res, "e2e": {"value": res["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                                          "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def e2e_run(R, wl, steps, stream, barrier, reduce_fn=None):
    """The same step through the public API with host buffers: every step
    copies its inputs (x, dy) from pinned host memory to the device and its
    results (the weight gradients dw and the data gradient dx of a training
    step, y of an inference step) back to pinned host memory, all inside the
    timed region.  The copies of step i+1's inputs and of step i's results run
    on a copy stream while step i+1 computes (inputs and results are double
    buffered on the device), ordered by events."""
    train = wl.training
    ins = ["x"] + (["dy"] if train else [])
    outs = ["dw", "dx"] if train else ["y"]
    dev_in = {k: [getattr(R, k), torch.empty_like(getattr(R, k))] for k in ins}
    for k in ins:
        dev_in[k][1].copy_(dev_in[k][0])
    dev_out = {k: [getattr(R, k), torch.empty_like(getattr(R, k))] for k in outs}
    host_in = {k: [torch.empty(dev_in[k][0].shape, dtype=dev_in[k][0].dtype, pin_memory=True) for _ in range(2)]
               for k in ins}
    for k in ins:
        for j in range(2):
            host_in[k][j].copy_(dev_in[k][0])
    host_out = {k: [torch.empty(dev_out[k][0].shape, dtype=dev_out[k][0].dtype, pin_memory=True) for _ in range(2)]
                for k in outs}
    h2d = sum(v[0].numel() * v[0].element_size() for v in dev_in.values())
    d2h = sum(v[0].numel() * v[0].element_size() for v in dev_out.values())
    cs = torch.cuda.Stream(device=stream.device)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer j landed
    ev_done = [torch.cuda.Event() for _ in range(2)]  # step on buffer j finished (inputs free, results ready)
    ev_out = [torch.cuda.Event() for _ in range(2)]   # results of buffer j copied out

    def bind(j):
        for k in ins:
            setattr(R, k, dev_in[k][j])
        for k in outs:
            setattr(R, k, dev_out[k][j])

    def upload(j):
        with torch.cuda.stream(cs):
            cs.wait_event(ev_done[j])  # the previous step on buffer j has read its inputs
            for k in ins:
                dev_in[k][j].copy_(host_in[k][j], non_blocking=True)
            ev_in[j].record(cs)

    def download(j):
        with torch.cuda.stream(cs):
            cs.wait_event(ev_done[j])
            for k in outs:
                host_out[k][j].copy_(dev_out[k][j], non_blocking=True)
            ev_out[j].record(cs)

    def run(n):
        for j in range(2):
            ev_done[j].record(stream)
            ev_out[j].record(stream)
        upload(0)
        for i in range(n):
            j = i & 1
            if i + 1 < n:
                upload(1 - j)
            stream.wait_event(ev_in[j])
            stream.wait_event(ev_out[j])  # results of the step before last on buffer j are out
            bind(j)
            R.step()
            if reduce_fn is not None:
                reduce_fn(R)
            ev_done[j].record(stream)
            download(j)
        for j in range(2):
            stream.wait_event(ev_out[j])

    run(6)  # warm-up: both buffer sets through the graph cache
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(steps)
    e1.record(stream)
    barrier()
    bind(0)
    # the host link of this machine: one read-back of the same results with nothing else running
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for k in outs:
        host_out[k][0].copy_(dev_out[k][0], non_blocking=True)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_run.d2h_gbs = d2h / (f0.elapsed_time(f1) * 1e-3) / 1e9
    return e0.elapsed_time(e1) / steps, h2d, d2h


def weight_bytes_per_launch(wl):
    """Algorithmic bytes of one recurrent-step launch: the W_h it must read
    (G*H*H in the storage type).  The state it reads and writes (gates, c,
    h, carry, P) is reported beside it, not counted in the roofline."""
    return wl.G * wl.hidden * wl.hidden * (2 if wl.mode == 1 else 4)


def class_roofline(name, n, tot, wl, steps, pk, transposed, fused_point):
    """Roofline of one kernel class from its serialised CUDA-event timings:
    algorithmic flops (2*M*N*K) per launch against the burst bf16 tensor peak
    (each launch is timed on its own), and for the recurrent steps the W_h
    bytes per launch against the measured copy bandwidth; the slower bound
    binds."""
    cf = class_flops(wl)
    sec = tot * 1e-3 / n
    flops = cf.get(name, 0.0) * steps / n
    nbytes = weight_bytes_per_launch(wl) if name in ("fwd_step", "bwd_step") else 0.0
    t_tensor = flops / (pk["bf16_tflops"] * 1e12)
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    out = {"kernel": name, "launches_per_step": n // steps, "flops_per_launch": flops,
           "bytes_per_launch": nbytes, "ms_per_launch": 1e3 * sec,
           "tensor_frac": flops / sec / 1e12 / pk["bf16_tflops"]}
    if name in ("fwd_step", "bwd_step"):
        cb = class_bytes(wl, transposed, fused_point)
        out["state_bytes_per_launch"] = cb[name] * steps / n - nbytes if name in cb else None
    if nbytes and t_hbm > t_tensor:
        ach = nbytes / sec / 1e9
        out.update(bound="hbm", achieved=ach, peak=pk["hbm_gbs"], unit="GB/s", frac=ach / pk["hbm_gbs"],
                   peak_source=pk["source"] + " copy bandwidth")
    else:
        ach = flops / sec / 1e12
        out.update(bound="tensor", achieved=ach, peak=pk["bf16_tflops"], unit="TFLOP/s", frac=ach / pk["bf16_tflops"],
                   peak_source=pk["source"] + " bf16 burst (kernel timed alone)")
    return out


def roofline(prof, wl, steps, pk, transposed, fused_point=False):
    """The dominant kernel class (largest device time) and its roofline; the
    DRAM traffic per launch from the committed ncu capture of the same build."""
    cf = class_flops(wl)
    cand = [(k, v) for k, v in prof.items() if k in cf and v[0] > 0]
    if not cand:
        return None
    name, (n, tot) = max(cand, key=lambda kv: kv[1][1])
    r = class_roofline(name, n, tot, wl, steps, pk, transposed, fused_point)
    r["measured_in"] = "serialised profiling pass (see kernels_note)"
    r["traffic"] = NCU_TRAFFIC.get((wl.name, name))
    return r


def kernel_profile(wl, dev, args):
    """Per-kernel CUDA-event timings of the same workload in a separate pass:
    launches serialised on the caller's stream (no wavefront overlap, no graph)
    and queued behind a GPU sleep so that the host is ahead of the device and
    consecutive event pairs bracket back-to-back kernels."""
    from recurrent_neural_network_gb300 import rnn
    flags = rnn.FLAG_PROFILE | rnn.FLAG_NO_WAVEFRONT | rnn.FLAG_NO_GRAPH
    R = make_runner(wl, dev, flags=flags)
    R.step()
    torch.cuda.synchronize()
    R.r.profile(reset=True)
    steps = max(1, min(args.steps, 3))
    torch.cuda._sleep(int(2e8))  # ~0.1 s of device time while the host enqueues
    for _ in range(steps):
        R.step()
    torch.cuda.synchronize()
    prof = R.r.profile(reset=True)
    assert R.status() == 0
    return prof, steps


def smem_peak_gbs(mhz):
    """Aggregate shared-memory read bandwidth derived from the unit counts:
    152 SMs x 128 B/clk x SM clock."""
    return 152 * 128 * mhz * 1e6 / 1e9


def fp32_peak_tflops(mhz):
    """FFMA peak derived from the unit counts: 152 SMs x 128 fp32 lanes x 2 flop x SM clock."""
    return 152 * 128 * 2 * mhz * 1e6 / 1e12


def workload_roofline(wl, ms, pk, persistent, stacked=False):
    """Roofline of a whole step: the slower of (a) its GEMM flops at the
    tensor peak (sustained: the step is a long run of kernels; the FFMA peak
    for the fp32 mode) and (b) the recurrent weights it must read, once per
    recurrent step of every layer and direction (forward, and again in the
    backward pass of a training step), from HBM when streamed or from shared
    memory when the persistent recurrence keeps them on chip.  The stacked
    recurrences keep the weights in tensor memory, the tensor core's own
    operand store, with no bandwidth bound of their own: their step is held
    to the tensor peak (the weight bytes are reported as read on chip)."""
    mhz = pk.get("sm_max_mhz", 2070.0)
    fl = step_flops(wl)
    if wl.mode == 1:
        tpk, tsrc = pk["bf16_tflops_sustained"], pk["source"] + " bf16 sustained"
    else:
        tpk, tsrc = fp32_peak_tflops(mhz), "derived FFMA: 152 SMs x 128 lanes x 2 x %.0f MHz" % mhz
    passes = wl.T * wl.layers * wl.directions * (2 if wl.training else 1)
    wbytes = passes * weight_bytes_per_launch(wl)
    bw, bsrc = ((smem_peak_gbs(mhz), "derived: 152 SMs x 128 B/clk x %.0f MHz" % mhz) if persistent
                else (pk["hbm_gbs"], pk["source"] + " copy bandwidth"))
    t_t = fl / (tpk * 1e12)
    t_w = wbytes / (bw * 1e9)
    sec = ms * 1e-3
    if stacked:
        return {"bound": "tensor", "achieved": fl / sec / 1e12, "peak": tpk, "unit": "TFLOP/s", "frac": t_t / sec,
                "weight_bytes_per_step": wbytes, "weights": "tensor memory (read on chip)", "peak_source": tsrc}
    if t_w > t_t:
        return {"bound": "smem" if persistent else "hbm", "achieved": wbytes / sec / 1e9, "peak": bw, "unit": "GB/s",
                "frac": t_w / sec, "weight_bytes_per_step": wbytes, "peak_source": bsrc,
                "tensor_frac": fl / sec / 1e12 / tpk}
    return {"bound": "tensor" if wl.mode == 1 else "alu", "achieved": fl / sec / 1e12, "peak": tpk,
            "unit": "TFLOP/s", "frac": t_t / sec, "weight_bytes_per_step": wbytes, "peak_source": tsrc,
            "weight_frac": t_w / sec}


def make_runner(wl, dev, flags=0, chunk=0, rank=0, world=1):
    """A Runner of wl on dev with its synthetic inputs drawn on the device;
    with world > 1, this rank's shard of a global batch of world * wl.B
    sequences (same weights on every rank)."""
    from recurrent_neural_network_gb300 import dp, runner, synth
    R = runner.Runner(wl, device=dev, flags=flags, chunk=chunk)
    gw = dp.global_batch(wl, world)

    def t(what, dtype):
        v = synth.device_tensor(gw, what, dev, dtype)
        return v if (world == 1 or what == "w") else dp.shard(v, rank, world, dim=1)
    R.x = t("x", R.dt)
    R.w_user = t("w", R.dt)
    R.h0 = t("h0", R.dt)
    R.c0 = t("c0", torch.float32) if wl.cell == synth.CELL_LSTM else None
    R.dy = t("dy", R.dt) if wl.training else None
    R.pack()
    return R


def workload_probe(idx, dev, pk, steps=10, warmup=3):
    """One of the other benchmark workloads, timed with CUDA events over
    `steps` whole steps after `warmup` (same step as the headline: forward,
    BPTT, weight gradients, or the forward of an inference workload)."""
    from recurrent_neural_network_gb300 import synth
    wl = synth.WORKLOADS[idx]
    R = make_runner(wl, dev)
    for _ in range(warmup):
        R.step()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record()
        R.forward()
        ev[i][1].record()
        if wl.training:
            R.backward()
        ev[i][2].record()
        if wl.training:
            R.weights()
        ev[i][3].record()
    torch.cuda.synchronize()
    assert R.status() == 0
    ms = ev[0][0].elapsed_time(ev[-1][3]) / steps
    phases = {nm: statistics.mean(e[k].elapsed_time(e[k + 1]) for e in ev)
              for k, nm in enumerate(["fwd", "bwd_data", "bwd_weights"])}
    plan = R.r.describe()
    persistent = "recurrence=persistent" in plan
    stacked = "recurrence=stacked" in plan
    out = {"ms_per_step": ms, "tflops": step_flops(wl) / (ms * 1e-3) / 1e12,
           "timesteps_per_s": wl.T / (ms * 1e-3), "us_per_timestep": 1e3 * ms / wl.T,
           "training": wl.training, "dtype": "bf16" if wl.mode == 1 else "f32", "plan": plan, "phases_ms": phases,
           "roofline": workload_roofline(wl, ms, pk, persistent, stacked)}
    del R
    torch.cuda.empty_cache()
    return wl.name, out


def fp8_stash_probe(dev, pk, steps=5, warmup=2):
    """The fp8 stash of W_h (RNN_FLAG_FP8_STASH): a 1-layer LSTM, H=2048, B=4,
    T=1000 inference, whose bf16 W_h (32 MiB) is too large for the
    register-resident recurrence, timed with the persistent recurrence on the
    e4m3 stash (16 MiB in shared memory across the CTAs) and with streaming
    bf16 steps.  Roofline of the stash: its bytes read from shared memory once
    per timestep at the aggregate shared-memory bandwidth."""
    from recurrent_neural_network_gb300 import rnn, synth
    wl = synth.Workload("lstm_bf16_L1_T1000_B4_H2048_infer", synth.CELL_LSTM, 1, 1000, 4, 2048, 2048,
                        synth.MODE_BF16, forget_bias=1.0, training=False)
    out = {"workload": wl.name}
    for name, fl in (("fp8_stash_persistent", rnn.FLAG_FP8_STASH), ("bf16_streaming", 0)):
        R = make_runner(wl, dev, flags=fl)
        for _ in range(warmup):
            R.forward(False)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            R.forward(False)
        e1.record()
        torch.cuda.synchronize()
        assert R.status() == 0
        ms = e0.elapsed_time(e1) / steps
        out[name] = {"ms_per_call": ms, "us_per_timestep": 1e3 * ms / wl.T, "timesteps_per_s": wl.T / (ms * 1e-3),
                     "plan": R.r.describe()}
        del R
        torch.cuda.empty_cache()
    mhz = pk.get("sm_max_mhz", 2070.0)
    stash = wl.G * wl.hidden * wl.hidden  # e4m3 bytes
    roof_us = stash / (smem_peak_gbs(mhz) * 1e9) * 1e6
    us = out["fp8_stash_persistent"]["us_per_timestep"]
    out["fp8_stash_persistent"]["roofline"] = {
        "bound": "smem", "bytes_per_timestep": stash, "peak": smem_peak_gbs(mhz), "unit": "GB/s",
        "achieved": stash / (us * 1e-6) / 1e9, "frac": roof_us / us,
        "peak_source": "derived: 152 SMs x 128 B/clk x %.0f MHz" % mhz}
    out["speedup_vs_streaming"] = out["bf16_streaming"]["ms_per_call"] / out["fp8_stash_persistent"]["ms_per_call"]
    return out


def sweep(dev, steps=5, warmup=2, cells=(0, 1), batches=(1, 2, 4, 8, 16, 32, 64, 128, 256, 512),
          widths=(256, 512, 1024, 2048, 4096, 8192), layers=1, T=16):
    """Selector sweep: bf16 training steps (`layers` layers, T timesteps) over
    batch sizes and widths, timed with the library's own plan and with each
    recurrence variant forced (persistent, stacked, streaming transposed,
    streaming row-major), one JSON line per shape.  Places the planner's
    switches (persistent / stacked / streaming, step orientation) and shows
    how throughput moves with the batch at each width."""
    from recurrent_neural_network_gb300 import rnn, synth
    variants = [("default", 0), ("persistent", rnn.FLAG_FORCE_PERSISTENT), ("stacked", rnn.FLAG_FORCE_STACK),
                ("transposed", rnn.FLAG_FORCE_TRANSPOSED | rnn.FLAG_FORCE_STREAMING),
                ("row_major", rnn.FLAG_NO_TRANSPOSED | rnn.FLAG_FORCE_STREAMING)]
    for cell in cells:
        for H in widths:
            for B in batches:
                wl = synth.Workload(name=f"sweep_c{cell}_B{B}_H{H}", cell=cell, layers=layers, T=T, B=B, input=H,
                                    hidden=H, mode=synth.MODE_BF16, forget_bias=1.0, state_std=0.1)
                res, plan = {}, None
                for name, fl in variants:
                    try:
                        R = make_runner(wl, dev, flags=fl)
                    except rnn.RnnError:
                        continue
                    if name == "default":
                        plan = R.r.describe()
                    for _ in range(warmup):
                        R.step()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    for _ in range(steps):
                        R.step()
                    e1.record()
                    torch.cuda.synchronize()
                    assert R.status() == 0
                    res[name] = e0.elapsed_time(e1) / steps
                    del R
                    torch.cuda.empty_cache()
                fl = step_flops(wl)
                forced = {k: v for k, v in res.items() if k != "default"}
                best = min(forced, key=forced.get) if forced else None
                print(json.dumps({"sweep": {"cell": synth.CELL_NAMES[cell], "L": layers, "T": T, "B": B, "H": H},
                                  "ms": {k: round(v, 4) for k, v in res.items()},
                                  "tflops": {k: round(fl / (v * 1e-3) / 1e12, 2) for k, v in res.items()},
                                  "best_forced": best, "plan": plan}), flush=True)


def synth_tensor(wl, what, dev, dtype):
    from recurrent_neural_network_gb300 import synth
    return synth.device_tensor(wl, what, dev, dtype)


def ncu_steps(args):
    """A short program for ncu: --ncu-T timesteps (default 2) of one layer of
    the configured workload (forward, BPTT, weight gradients; the forward of an
    inference workload), run twice, no timing."""
    from recurrent_neural_network_gb300 import build, runner, synth
    build.build()
    dev = torch.device("cuda", 0)
    wl = synth.WORKLOADS[args.config].replace(layers=1, T=args.ncu_T)
    R = runner.Runner(wl, device=dev, flags=args.flags, chunk=args.chunk)
    R.x = synth_tensor(wl, "x", dev, R.dt)
    R.w_user = synth_tensor(wl, "w", dev, R.dt)
    R.h0 = synth_tensor(wl, "h0", dev, R.dt)
    if wl.cell == synth.CELL_LSTM:
        R.c0 = synth_tensor(wl, "c0", dev, torch.float32)
    R.dy = synth_tensor(wl, "dy", dev, R.dt) if wl.training else None
    R.pack()
    for _ in range(2):
        R.step()
    torch.cuda.synchronize()
    assert R.status() == 0
    print(json.dumps({"ncu_steps": wl.name, "plan": R.r.describe()}))


def one_step(args):
    """One direct training step (forward, BPTT, weight gradients) of workload
    --config with its default plan, after packing the weights: the launch
    list of a profiler run over it is one step's kernels.  Prints the device
    status word (0, or the error code a kernel recorded) and the plan."""
    from recurrent_neural_network_gb300 import build, rnn, synth
    build.build()
    wl = synth.WORKLOADS[args.config]
    R = make_runner(wl, torch.device("cuda", 0), flags=args.flags | rnn.FLAG_NO_GRAPH, chunk=args.chunk)
    R.step()
    torch.cuda.synchronize()
    print(json.dumps({"one_step": wl.name, "status": R.status(), "plan": R.r.describe()}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the sub-results of the other workloads")
    ap.add_argument("--flags", type=int, default=0)
    ap.add_argument("--chunk", type=int, default=0)
    ap.add_argument("--sweep", action="store_true",
                    help="selector sweep over batch sizes and widths instead of the benchmark line")
    ap.add_argument("--sweep-shape", default="1,16",
                    help="layers,timesteps of the sweep's training steps (e.g. 4,100 for the stacked range)")
    ap.add_argument("--sweep-batches", default="1,2,4,8,16,32,64,128,256,512")
    ap.add_argument("--sweep-widths", default="256,512,1024,2048,4096,8192")
    ap.add_argument("--sweep-cells", default="0,1", help="cells of the sweep (0 LSTM, 1 GRU, 2 tanh, 3 ReLU)")
    ap.add_argument("--one-step", action="store_true",
                    help="one direct training step of the --config workload (packing included), for launch lists")
    ap.add_argument("--ncu-T", type=int, default=2, help="timesteps of the --ncu-steps program")
    ap.add_argument("--ncu-steps", action="store_true",
                    help="one training pass (forward, BPTT, weight gradients) of a one-layer T=2 copy of the "
                         "workload, for profiler captures: every recurrent-step launch has the full per-step shape")
    args = ap.parse_args()
    if args.sweep:
        from recurrent_neural_network_gb300 import build
        build.build()
        layers, T = (int(v) for v in args.sweep_shape.split(","))
        sweep(torch.device("cuda", 0), layers=layers, T=T, cells=tuple(int(v) for v in args.sweep_cells.split(",")),
              batches=tuple(int(v) for v in args.sweep_batches.split(",")),
              widths=tuple(int(v) for v in args.sweep_widths.split(",")))
        return
    if args.ncu_steps:
        ncu_steps(args)
        return
    if args.one_step:
        one_step(args)
        return

    from recurrent_neural_network_gb300 import synth
    wl = synth.WORKLOADS[args.config]
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, wl, rank)
        return

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from recurrent_neural_network_gb300 import build, dp, rnn
    build.build()
    dev = torch.device("cuda", local)
    R = make_runner(wl, dev, flags=args.flags, chunk=args.chunk, rank=rank, world=world)
    torch.cuda.synchronize()
    # data-parallel exchange: dW summed over the ranks once per training step
    reduce_fn = (lambda r: dp.allreduce_grads_(r.dw)) if (world > 1 and wl.training) else None

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        R.step()
        if reduce_fn is not None:
            reduce_fn(R)
    assert R.status() == 0

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    clocks = Clocks(local)
    barrier()
    clocks.start()
    time.sleep(0.25)
    n_launch0 = rnn.launch_count()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for i in range(args.steps):
        # phase boundaries on the caller's stream: forward | BPTT | weight gradients | dW all-reduce
        ev[i][0].record(stream)
        R.forward()
        ev[i][1].record(stream)
        if wl.training:
            R.backward()
        ev[i][2].record(stream)
        if wl.training:
            R.weights()
        ev[i][3].record(stream)
        if reduce_fn is not None:
            reduce_fn(R)
        ev[i][4].record(stream)
    barrier()
    launches = rnn.launch_count() - n_launch0
    ms = ev[0][0].elapsed_time(ev[-1][4]) / args.steps
    phases = {nm: statistics.mean(e[k].elapsed_time(e[k + 1]) for e in ev)
              for k, nm in enumerate(["fwd", "bwd_data", "bwd_weights", "dw_allreduce"])}
    clk = clocks.stop()
    st = R.status()
    assert st == 0, f"device status {st}"
    fl = step_flops(wl)
    ms, tflops, world = replica_aggregate(ms, fl, dist, dev)
    pk = peaks()
    e2e_clk = None
    if args.no_e2e:
        ms_e2e, h2d, d2h = float("nan"), 0, 0
    else:
        clocks_e2e = Clocks(local)
        clocks_e2e.start()
        ms_e2e, h2d, d2h = e2e_run(R, wl, args.steps, stream, barrier, reduce_fn)
        e2e_clk = clocks_e2e.stop()
        ms_e2e, _, _ = replica_aggregate(ms_e2e, fl, dist, dev)
    plan = R.r.describe()
    del R
    torch.cuda.empty_cache()
    prof, psteps = kernel_profile(wl, dev, args)
    roof = roofline(prof, wl, psteps, pk, "transposed=1" in plan, "fused_point=1" in plan)
    subs = {}
    if world == 1 and not args.no_workloads:
        for idx in range(5):
            if idx != args.config:
                name, res = workload_probe(idx, dev, pk)
                subs[name] = res

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if wl.mode == 1 else "f32", "data": "synthetic",
        "timesteps_per_s": world * wl.T / (ms * 1e-3),
        "tensor_peak_frac": {"of_measured_burst": tflops / world / pk["bf16_tflops"],
                             "of_measured_sustained": tflops / world / pk["bf16_tflops_sustained"]},
        "config": {"workload": wl.name, "cell": synth.CELL_NAMES[wl.cell], "layers": wl.layers, "T": wl.T,
                   "B": wl.B, "global_batch": wl.B * world, "input": wl.input, "hidden": wl.hidden,
                   "training": wl.training, "flops_per_step": fl, "plan": plan,
                   "parallelism": f"dp{world}" if world > 1 else "single",
                   "dp_exchange": "NCCL all-reduce (sum) of dW every step" if reduce_fn is not None else None,
                   "l2": "inputs larger than L2 (weights, reserve and activations exceed 129 MB)"},
        "gpu_launches": launches,
        "roofline": roof,
        "step_roofline": workload_roofline(wl, ms, pk, "recurrence=persistent" in plan),
        "clocks": clk,
        "e2e": {"value": world * fl / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                "d2h_gbs_alone": None if args.no_e2e else round(getattr(e2e_run, "d2h_gbs", float("nan")), 1),
                "clocks": e2e_clk,
                "copies": ("x, dy in; dw, dx out" if wl.training else "x in; y out") +
                          ", pinned host buffers, overlapped with the neighbouring steps on a copy stream; "
                          "d2h_gbs_alone: one read-back of the same results with nothing else running"},
        "phases_ms": phases,
        "workloads": subs,
        "kernels": {k: class_roofline(k, v[0], v[1], wl, psteps, pk, "transposed=1" in plan, "fused_point=1" in plan)
                    for k, v in prof.items() if v[0] and k in class_flops(wl)},
        "kernels_note": "per-kernel CUDA-event times from a separate pass of the same workload with launches "
                        "serialised (no wavefront, no graph); the timed run overlaps layers and replays graphs",
        # every kernel class of that pass (the stacked and persistent recurrences included, which ncu
        # cannot time: it launches them without their cluster shape): launches and ms per step
        "kernel_classes": {k: {"launches": v[0] // psteps, "ms": round(v[1] / psteps, 4)}
                           for k, v in sorted(prof.items()) if v[0]},
    }
    # the persistent small-batch recurrence (second target of the path) under its own key as well
    line["persistent_recurrence"] = subs.get(synth.WORKLOADS[2].name)
    if world == 1 and not args.no_workloads:
        line["fp8_stash"] = fp8_stash_probe(dev, pk)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"], _ = time_oracle_sample(wl)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
