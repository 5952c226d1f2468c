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
products), with timesteps/s beside it.  With N > 1 (torchrun) every rank runs
an independent replica of the workload (no collective on the data path).
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
        sm, mx, reasons = [], [], set()
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
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


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
# product); summarised in profiles/ncu_step_kernels_lstm_B256_H4096.md.
NCU_TRAFFIC = {("lstm_bf16_L4_T50_B256_H4096", "bwd_step"): 177.36e6,
               ("lstm_bf16_L4_T50_B256_H4096", "fwd_step"): 162.64e6}


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


def e2e_run(R, wl, steps, sdt, stream, barrier):
    """The same step through the public API with the inputs in pinned host
    memory: host->device copies of x (and dy) and a device->host read of hT
    inside the timed region."""
    hx = torch.empty(R.x.shape, dtype=sdt, pin_memory=True)
    hx.copy_(R.x)
    hdy = None
    if wl.training:
        hdy = torch.empty(R.dy.shape, dtype=sdt, pin_memory=True)
        hdy.copy_(R.dy)
    hout = torch.empty(R.hT.shape, dtype=R.hT.dtype, pin_memory=True)
    h2d = hx.numel() * hx.element_size() + (hdy.numel() * hdy.element_size() if hdy is not None else 0)
    d2h = hout.numel() * hout.element_size()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        R.x.copy_(hx, non_blocking=True)
        if hdy is not None:
            R.dy.copy_(hdy, non_blocking=True)
        R.step()
        hout.copy_(R.hT, non_blocking=True)
    e1.record(stream)
    barrier()
    return e0.elapsed_time(e1) / steps, h2d, d2h


def roofline(prof, wl, steps, pk, transposed, fused_point=False):
    """Roofline of the dominant kernel class (largest device time): its
    algorithmic flops and bytes per launch over its average CUDA-event launch
    duration, against the tensor or the HBM peak, whichever its arithmetic
    intensity makes binding."""
    cf, cb = class_flops(wl), class_bytes(wl, transposed, fused_point)
    cand = [(k, v) for k, v in prof.items() if k in cf and v[0] > 0]
    if not cand:
        return None
    name, (n, tot) = max(cand, key=lambda kv: kv[1][1])
    sec = tot * 1e-3 / n
    flops = cf[name] * steps / n
    t_tensor = flops / (pk["bf16_tflops_sustained"] * 1e12)
    nbytes = cb[name] * steps / n if name in cb else 0.0
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9) if nbytes else 0.0
    common = {"kernel": name, "launches_per_step": n // steps, "flops_per_launch": flops, "bytes_per_launch": nbytes,
              "ms_per_launch": 1e3 * sec, "measured_in": "serialised profiling pass (see kernels_note)",
              "traffic": NCU_TRAFFIC.get((wl.name, name))}
    if t_hbm > t_tensor:
        ach = nbytes / sec / 1e9
        return dict(common, bound="hbm", achieved=ach, peak=pk["hbm_gbs"], unit="GB/s", frac=ach / pk["hbm_gbs"],
                    tensor_frac=flops / sec / 1e12 / pk["bf16_tflops_sustained"],
                    peak_source=pk["source"] + " (copy bandwidth)")
    ach = flops / sec / 1e12
    return dict(common, bound="tensor", achieved=ach, peak=pk["bf16_tflops_sustained"], unit="TFLOP/s",
                frac=ach / pk["bf16_tflops_sustained"],
                peak_source=pk["source"] + " (sustained bf16, kernel timed inside the step)")


def kernel_profile(wl, dev, args, sdt):
    """Per-kernel CUDA-event timings of the same workload in a separate pass:
    launches serialised on the caller's stream (no wavefront overlap, no graph)
    and queued behind a GPU sleep so that the host is ahead of the device and
    consecutive event pairs bracket back-to-back kernels."""
    from recurrent_neural_network_gb300 import rnn, runner
    flags = rnn.FLAG_PROFILE | rnn.FLAG_NO_WAVEFRONT | rnn.FLAG_NO_GRAPH
    R = runner.Runner(wl, device=dev, flags=flags)
    R.x = synth_tensor(wl, "x", dev, sdt)
    R.w_user = synth_tensor(wl, "w", dev, sdt)
    R.h0 = synth_tensor(wl, "h0", dev, sdt)
    R.c0 = synth_tensor(wl, "c0", dev, torch.float32) if wl.cell == 0 else None
    R.dy = synth_tensor(wl, "dy", dev, sdt) if wl.training else None
    R.pack()
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


def persistent_probe(dev, steps=10, warmup=3):
    """Second target of the path: the persistent small-batch recurrence
    (1-layer LSTM, B=4, H=1024, T=1000 inference).  Per step it reads the
    8 MiB W_h from on-chip storage; its roofline is that read at the
    aggregate shared-memory bandwidth of the GPU, derived from the unit
    counts (152 SMs x 128 B/clk x max SM clock)."""
    from recurrent_neural_network_gb300 import rnn, runner, synth
    wl = synth.WORKLOADS[2]
    R = runner.Runner(wl, device=dev, flags=rnn.FLAG_FORCE_PERSISTENT)
    R.x = synth_tensor(wl, "x", dev, R.dt)
    R.w_user = synth_tensor(wl, "w", dev, R.dt)
    R.h0 = synth_tensor(wl, "h0", dev, R.dt)
    R.c0 = synth_tensor(wl, "c0", dev, torch.float32)
    R.pack()
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
    pk = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    mhz = pk.get("sm_max_mhz", 2070.0)
    smem_gbs = 152 * 128 * mhz * 1e6 / 1e9
    wh_bytes = 4 * wl.hidden * wl.hidden * 2
    us_step = 1e3 * ms / wl.T
    roof_us = wh_bytes / (smem_gbs * 1e9) * 1e6
    return {"workload": wl.name, "ms_per_call": ms, "us_per_timestep": us_step, "timesteps_per_s": wl.T / (ms * 1e-3),
            "tflops": step_flops(wl) / (ms * 1e-3) / 1e12, "plan": R.r.describe(),
            "roofline": {"bound": "smem", "bytes_per_timestep": wh_bytes, "peak": smem_gbs, "unit": "GB/s",
                         "peak_source": "derived: 152 SMs x 128 B/clk x %.0f MHz" % mhz,
                         "roofline_us_per_timestep": roof_us, "achieved": wh_bytes / (us_step * 1e-6) / 1e9,
                         "frac": roof_us / us_step}}


def sweep(dev, steps=5, warmup=2):
    """Selector sweep: one-layer bf16 LSTM and tanh-RNN training steps (T=16)
    over a grid of batch sizes and widths, timed with the library's own plan
    and with each recurrent-step orientation forced, one JSON line per shape.
    Used to place the planner's switch between the two orientations."""
    from recurrent_neural_network_gb300 import rnn, runner, synth
    variants = [("default", 0), ("transposed", rnn.FLAG_FORCE_TRANSPOSED | rnn.FLAG_FORCE_STREAMING),
                ("row_major", rnn.FLAG_NO_TRANSPOSED | rnn.FLAG_FORCE_STREAMING)]
    for cell, H, B in [(c, h, b) for c in (0, 2) for h in (512, 1024, 2048, 4096) for b in (16, 32, 64, 128, 256)]:
        if True:
            wl = synth.Workload(name=f"sweep_c{cell}_B{B}_H{H}", cell=cell, layers=1, T=16, B=B, input=H, hidden=H,
                                mode=synth.MODE_BF16, forget_bias=1.0, state_std=0.1)
            res, plan = {}, None
            for name, fl in variants:
                try:
                    R = runner.Runner(wl, device=dev, flags=fl)
                except rnn.RnnError:
                    continue
                if name == "default":
                    plan = R.r.describe()
                R.x = synth_tensor(wl, "x", dev, R.dt)
                R.w_user = synth_tensor(wl, "w", dev, R.dt)
                R.h0 = synth_tensor(wl, "h0", dev, R.dt)
                R.c0 = synth_tensor(wl, "c0", dev, torch.float32) if cell == 0 else None
                R.dy = synth_tensor(wl, "dy", dev, R.dt)
                R.pack()
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
            print(json.dumps({"sweep": {"cell": ["lstm", "gru", "tanh"][cell], "L": 1, "T": 16, "B": B, "H": H},
                              "ms": {k: round(v, 4) for k, v in res.items()},
                              "tflops": {k: round(fl / (v * 1e-3) / 1e12, 1) for k, v in res.items()},
                              "plan": plan}), flush=True)


def synth_tensor(wl, what, dev, dtype):
    from recurrent_neural_network_gb300 import synth
    return synth.device_tensor(wl, what, dev, dtype)


def ncu_steps(args):
    """A short program for ncu: two timesteps of one layer of the configured
    workload (forward, BPTT, weight gradients), run twice, no timing."""
    from recurrent_neural_network_gb300 import build, runner, synth
    build.build()
    dev = torch.device("cuda", 0)
    wl = synth.WORKLOADS[args.config].replace(layers=1, T=2)
    R = runner.Runner(wl, device=dev, flags=args.flags, chunk=args.chunk)
    R.x = synth_tensor(wl, "x", dev, R.dt)
    R.w_user = synth_tensor(wl, "w", dev, R.dt)
    R.h0 = synth_tensor(wl, "h0", dev, R.dt)
    if wl.cell == synth.CELL_LSTM:
        R.c0 = synth_tensor(wl, "c0", dev, torch.float32)
    R.dy = synth_tensor(wl, "dy", dev, R.dt)
    R.pack()
    for _ in range(2):
        R.step()
    torch.cuda.synchronize()
    assert R.status() == 0
    print(json.dumps({"ncu_steps": wl.name, "plan": R.r.describe()}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-persistent", action="store_true")
    ap.add_argument("--flags", type=int, default=0)
    ap.add_argument("--chunk", type=int, default=0)
    ap.add_argument("--sweep", action="store_true",
                    help="selector sweep over batch sizes and widths instead of the benchmark line")
    ap.add_argument("--ncu-steps", action="store_true",
                    help="one training pass (forward, BPTT, weight gradients) of a one-layer T=2 copy of the "
                         "workload, for profiler captures: every recurrent-step launch has the full per-step shape")
    args = ap.parse_args()
    if args.sweep:
        from recurrent_neural_network_gb300 import build
        build.build()
        sweep(torch.device("cuda", 0))
        return
    if args.ncu_steps:
        ncu_steps(args)
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

    from recurrent_neural_network_gb300 import build, rnn, runner
    build.build()
    dev = torch.device("cuda", local)
    R = runner.Runner(wl, device=dev, flags=args.flags, chunk=args.chunk)
    sdt = R.dt
    R.x = synth.device_tensor(wl, "x", dev, sdt)
    R.w_user = synth.device_tensor(wl, "w", dev, sdt)
    R.h0 = synth.device_tensor(wl, "h0", dev, sdt)
    R.c0 = synth.device_tensor(wl, "c0", dev, torch.float32) if wl.cell == synth.CELL_LSTM else None
    R.dy = synth.device_tensor(wl, "dy", dev, sdt) if wl.training else None
    R.pack()
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        R.step()
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
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for i in range(args.steps):
        # phase boundaries on the caller's stream: forward | BPTT | weight gradients
        ev[i][0].record(stream)
        R.forward()
        ev[i][1].record(stream)
        if wl.training:
            R.backward()
        ev[i][2].record(stream)
        if wl.training:
            R.weights()
        ev[i][3].record(stream)
    barrier()
    launches = rnn.launch_count() - n_launch0
    ms = ev[0][0].elapsed_time(ev[-1][3]) / args.steps
    phases = {nm: statistics.mean(e[k].elapsed_time(e[k + 1]) for e in ev)
              for k, nm in enumerate(["fwd", "bwd_data", "bwd_weights"])}
    clk = clocks.stop()
    st = R.status()
    assert st == 0, f"device status {st}"
    fl = step_flops(wl)
    ms, tflops, world = replica_aggregate(ms, fl, dist, dev)
    pk = peaks()
    if args.no_e2e:
        ms_e2e, h2d, d2h = float("nan"), 0, 0
    else:
        ms_e2e, h2d, d2h = e2e_run(R, wl, args.steps, sdt, stream, barrier)
    plan = R.r.describe()
    del R
    torch.cuda.empty_cache()
    prof, psteps = kernel_profile(wl, dev, args, sdt)
    roof = roofline(prof, wl, psteps, pk, "transposed=1" in plan, "fused_point=1" in plan)
    persistent = persistent_probe(dev) if (world == 1 and args.config != 2 and not args.no_persistent) else None

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
                   "B": wl.B, "input": wl.input, "hidden": wl.hidden, "training": wl.training,
                   "flops_per_step": fl, "plan": plan,
                   "l2": "inputs larger than L2 (weights, reserve and activations exceed 129 MB)"},
        "gpu_launches": launches,
        "roofline": roof,
        "clocks": clk,
        "e2e": {"value": world * fl / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e},
        "phases_ms": phases,
        "persistent_recurrence": persistent,
        "kernels": {k: {"launches": v[0] // psteps, "ms_per_step": v[1] / psteps, "us_per_launch": 1e3 * v[1] / v[0]}
                    for k, v in prof.items() if v[0]},
        "kernels_note": "per-kernel CUDA-event times from a separate pass of the same workload with launches "
                        "serialised (no wavefront, no graph); the timed run overlaps layers and replays graphs",
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"], _ = time_oracle_sample(wl)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
