"""Helpers shared by the GPU parity tests: run the CUDA path through the C-ABI
and the oracle on the same seeded inputs, and compare them with the stated
tolerances.

Tolerances (fixed by the benchmark definition of this path):
  fp32 storage mode: max relative error <= 1e-4 on every output, with the
    relative error of element i taken as |g_i - o_i| / max(|o_i|, 1e-3 max_j |o_j|)
    per output tensor (the benchmark definition states no floor; one is needed
    where outputs pass through zero, and 1e-3 of the tensor's largest magnitude
    is the reading taken);
  bf16 storage mode: max absolute error <= 3e-2 on y, hT and cT, and relative
    L2 error ||g - o|| / ||o|| <= 2e-2 on dx, dh0, dc0 and each weight /
    bias gradient block.
"""
import numpy as np

import oracle
from recurrent_neural_network_gb300 import runner, synth

FP32_MAX_REL = 1e-4
FP32_FLOOR = 1e-3
BF16_MAX_ABS = 3e-2
BF16_REL_L2 = 2e-2


def kernel_decisions(wl):
    """Precision in which the ReLU cell's on/off decisions are taken on the
    oracle side: the one the device stores h in (bf16 or fp32).  Where a
    floating-point value decides a discrete choice, both sides take it in the
    kernel's precision; every value stays double."""
    return (1 if wl.mode == synth.MODE_BF16 else 2) if wl.cell == synth.CELL_RELU else 0


def run_oracle(hi: runner.HostInputs, train=True, lens=None, decide=None, on=None):
    w = hi.wl
    decide = kernel_decisions(w) if decide is None else decide
    y, hT, cT = oracle.fwd(w.cell, w.layers, w.T, w.B, w.input, w.hidden, hi.x, hi.w, h0=hi.h0, c0=hi.c0, lens=lens,
                           D=w.directions, decide=decide, on=on)
    out = dict(y=y, hT=hT, cT=cT)
    if train:
        dx, dh0, dc0, dw = oracle.bwd(w.cell, w.layers, w.T, w.B, w.input, w.hidden, hi.x, hi.w, hi.dy, h0=hi.h0,
                                      c0=hi.c0, dhT=hi.dhT, dcT=hi.dcT, lens=lens, D=w.directions, decide=decide,
                                      on=on)
        out.update(dx=dx, dh0=dh0, dc0=dc0, dw=dw)
    return out


def run_gpu(wl, hi, flags=0, chunk=0, train=None, timeout_ns=0, repeat=1, lens=None):
    r = runner.Runner(wl, flags=flags, chunk=chunk, timeout_ns=timeout_ns)
    if lens is not None:
        r.r.set_lengths(lens)
    r.upload(hi)
    train = wl.training if train is None else train
    for _ in range(repeat):
        if train:
            r.forward(True)
            r.backward()
            r.weights()
        else:
            r.forward(False)
    st = r.status()
    assert st == 0, f"device status {st}"
    return r.outputs()


def max_rel(g, o):
    g = np.asarray(g, np.float64).ravel()
    o = np.asarray(o, np.float64).ravel()
    floor = FP32_FLOOR * max(np.abs(o).max(), 1e-30)
    return float((np.abs(g - o) / np.maximum(np.abs(o), floor)).max())


def rel_l2(g, o):
    g = np.asarray(g, np.float64).ravel()
    o = np.asarray(o, np.float64).ravel()
    n = np.linalg.norm(o)
    return float(np.linalg.norm(g - o) / n) if n > 0 else float(np.linalg.norm(g))


def weight_blocks(wl, dw):
    """(name, array) per layer and part of a user-layout gradient vector."""
    out = []
    for l, parts in enumerate(oracle.split_weights(wl.cell, wl.layers, wl.input, wl.hidden, dw, D=wl.directions)):
        for nm, a in zip(("dWx", "dWh", "dbx", "dbh"), parts):
            out.append((f"l{l}.{nm}", a))
    return out


def compare(wl, g, o, keys=None, report=None):
    """Assert parity of every output both sides produced; returns the error table."""
    errs = {}
    keys = keys or [k for k in ("y", "hT", "cT", "dx", "dh0", "dc0") if o.get(k) is not None and g.get(k) is not None]
    for k in keys:
        if wl.mode == synth.MODE_FP32:
            errs[k] = ("max_rel", max_rel(g[k], o[k]), FP32_MAX_REL)
        elif k in ("y", "hT", "cT"):
            errs[k] = ("max_abs", float(np.abs(g[k] - o[k]).max()), BF16_MAX_ABS)
        else:
            errs[k] = ("rel_l2", rel_l2(g[k], o[k]), BF16_REL_L2)
    if g.get("dw") is not None and o.get("dw") is not None:
        for (nm, ga), (_, oa) in zip(weight_blocks(wl, g["dw"]), weight_blocks(wl, o["dw"])):
            if not np.any(oa) and not np.any(ga):
                continue
            if wl.mode == synth.MODE_FP32:
                errs[nm] = ("max_rel", max_rel(ga, oa), FP32_MAX_REL)
            else:
                errs[nm] = ("rel_l2", rel_l2(ga, oa), BF16_REL_L2)
    if report is not None:
        report.update(errs)
    bad = {k: v for k, v in errs.items() if not (v[1] <= v[2])}
    assert not bad, f"parity failed: {bad}"
    return errs


def sub_inputs(hi, layers):
    """The host inputs of the first `layers` layers of a stack (weights are
    stored layer by layer, so the first layers' weights are a prefix)."""
    wl = hi.wl.replace(layers=layers)
    out = object.__new__(type(hi))
    out.__dict__.update(hi.__dict__)
    out.wl = wl
    out.w = hi.w[:wl.weight_count()]
    out.h0 = hi.h0[:wl.states]
    out.c0 = None if hi.c0 is None else hi.c0[:wl.states]
    out.dhT = None if hi.dhT is None else hi.dhT[:wl.states]
    out.dcT = None if hi.dcT is None else hi.dcT[:wl.states]
    return out


def device_relu_decisions(wl, hi, g, flags=0, chunk=0, lens=None, cols=None):
    """The on/off decision of every ReLU unit as the device took it, [L*D][T][B][H]:
    on where its output h > 0.  Layer l's outputs come from an (l+1)-layer run
    of the same inputs, which computes the first l+1 layers exactly as the full
    stack does (same kernels and plan per layer); the top layer's from g.
    cols: restrict to these batch columns."""
    L, D, H = wl.layers, wl.directions, wl.hidden
    on = []
    for l in range(L):
        y = g["y"] if l == L - 1 else run_gpu(wl.replace(layers=l + 1), sub_inputs(hi, l + 1), flags=flags,
                                               chunk=chunk, lens=lens)["y"]
        if cols is not None:
            y = y[:, cols]
        for d in range(D):
            on.append((y[:, :, d * H:(d + 1) * H] > 0).astype(np.uint8))
    return np.stack(on)


def relu_check(wl, hi, g, on_dev, lens=None):
    """Parity of a ReLU run with the decisions the device took.  Each decision
    that differs from the oracle's (taken in the device's storage precision)
    must sit at a pre-activation within the forward bar of 0 (there the device's
    own pre-activation may lie on the other side of 0 within the stated
    tolerance); the outputs and gradients must then match the oracle computed
    with the device's decisions.  Returns the number of differing decisions."""
    on_ref, pre = oracle.relu_decisions(wl.layers, wl.T, wl.B, wl.input, wl.hidden, hi.x, hi.w, h0=hi.h0,
                                        lens=lens, D=wl.directions, decide=kernel_decisions(wl))
    diff = on_dev != on_ref
    far = np.abs(pre[diff]) > (BF16_MAX_ABS if wl.mode == synth.MODE_BF16 else 1e-4)
    assert not far.any(), f"{int(far.sum())} decisions differ away from the kink: |a| up to {np.abs(pre[diff]).max()}"
    compare(wl, g, run_oracle(hi, lens=lens, decide=3, on=on_dev))
    return int(diff.sum())
