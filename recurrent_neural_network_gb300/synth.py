"""Seeded synthetic inputs for the stacked-RNN workloads.

This module only draws numbers. It holds none of the recurrent arithmetic:
both the CUDA path and the double-precision oracle receive the arrays it
produces, so they see identical inputs.

Generator: counter-based splitmix64.  Element ``i`` of tensor ``tid`` under
seed ``s`` is the (i+1)-th output of a splitmix64 stream keyed by
``mix(mix(s) ^ tid)``.  Any slice (a prefix of timesteps, one batch column)
therefore regenerates identically without drawing the rest.  Uniforms are the
top 53 bits scaled to [0, 1); normals use the Box-Muller transform on the
uniforms of counters ``2i`` and ``2i+1``.

Workload recipes follow the sizes and distributions stated for the five
benchmark cases (one tiny fp32 LSTM, a 4-layer H=512 LSTM, a B=4 H=1024
inference LSTM, a 4-layer H=4096 B=256 LSTM and an 8-layer H=1024 GRU).  The
pages behind the method ("Optimizing Performance of Recurrent Neural Networks
on GPUs", review page, section "주요 결과") measure only throughput on
unnamed network sizes; these recipes stand in for those networks.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

_GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

CELL_LSTM, CELL_GRU, CELL_TANH, CELL_RELU = 0, 1, 2, 3
CELL_NAMES = {CELL_LSTM: "lstm", CELL_GRU: "gru", CELL_TANH: "tanh", CELL_RELU: "relu"}
GATES = {CELL_LSTM: 4, CELL_GRU: 3, CELL_TANH: 1, CELL_RELU: 1}
MODE_FP32, MODE_BF16 = 0, 1

# tensor ids of the counter streams
TID_X, TID_H0, TID_C0, TID_DY, TID_DHT, TID_DCT = 1, 3, 4, 5, 6, 7


def _s64(v: int) -> int:
    """Two's-complement int64 with the same 64 bits as the unsigned value v."""
    v &= (1 << 64) - 1
    return v - (1 << 64) if v >= (1 << 63) else v


def _mix_int(z: int) -> int:
    m = (1 << 64) - 1
    z = ((z ^ (z >> 30)) * _M1) & m
    z = ((z ^ (z >> 27)) * _M2) & m
    return z ^ (z >> 31)


def _key(seed: int, tid: int) -> int:
    m = (1 << 64) - 1
    k = _mix_int((seed + _GAMMA) & m)
    return _mix_int(((k ^ tid) + _GAMMA) & m)


def _srl(z, k):
    """Logical right shift of int64 tensors holding uint64 bit patterns."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def _uniform_bits(key: int, start: int, count: int, device):
    # int64 arithmetic wraps modulo 2^64 exactly like uint64
    idx = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    z = idx * _s64(_GAMMA) + _s64(key)
    z = (z ^ _srl(z, 30)) * _s64(_M1)
    z = (z ^ _srl(z, 27)) * _s64(_M2)
    z = z ^ _srl(z, 31)
    return _srl(z, 11)  # top 53 bits


def uniform01_t(seed: int, tid: int, start: int, count: int, device="cpu"):
    """U[0,1) float64 tensor for counters start .. start+count-1."""
    return _uniform_bits(_key(seed, tid), start, count, device).to(torch.float64) * (1.0 / 9007199254740992.0)


def uniform01(seed: int, tid: int, start: int, count: int) -> np.ndarray:
    return uniform01_t(seed, tid, start, count).numpy()


def uniform_t(seed, tid, shape, lo, hi, device="cpu"):
    n = int(np.prod(shape))
    return (lo + (hi - lo) * uniform01_t(seed, tid, 0, n, device)).reshape(shape)


def normal_t(seed, tid, shape, std=1.0, device="cpu"):
    n = int(np.prod(shape))
    u = uniform01_t(seed, tid, 0, 2 * n, device)
    u1, u2 = u[0::2], u[1::2]
    r = torch.sqrt(-2.0 * torch.log1p(-u1))
    return (std * r * torch.cos(2.0 * math.pi * u2)).reshape(shape)


def uniform(seed, tid, shape, lo, hi):
    return uniform_t(seed, tid, shape, lo, hi).numpy()


def normal(seed, tid, shape, std=1.0):
    return normal_t(seed, tid, shape, std).numpy()


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, storage mode and input distributions."""
    name: str
    cell: int
    layers: int
    T: int
    B: int
    input: int
    hidden: int
    mode: int
    x_dist: str = "normal"        # "normal" N(0,1) or "uniform" U(-1,1)
    forget_bias: float = 0.0      # added to b_x of the LSTM forget gate
    state_std: float = 0.0        # h0 (and c0) ~ N(0, state_std^2); 0 means zeros
    training: bool = True
    seed: int = 0
    # > 0: weights shrunk 20x and b_x = +kink_margin / -kink_margin on even /
    # odd units, so that every pre-activation of a ReLU RNN stays well away
    # from 0 and the activation's on/off decision is the same at any precision
    # (an option of the recipe; the workloads use the ordinary distribution)
    kink_margin: float = 0.0
    # 2: bidirectional layers (a second set of weights per layer runs time
    # backwards; outputs and the next layer's input are 2*hidden wide)
    directions: int = 1

    @property
    def G(self):
        return GATES[self.cell]

    def in_size(self, l):
        return self.input if l == 0 else self.directions * self.hidden

    def layer_weight_count(self, l):
        """Weights of one direction of layer l."""
        G, H = self.G, self.hidden
        return G * H * self.in_size(l) + G * H * H + 2 * G * H

    def weight_count(self):
        return sum(self.directions * self.layer_weight_count(l) for l in range(self.layers))

    @property
    def states(self):
        """Rows of the state arrays: one per (layer, direction)."""
        return self.layers * self.directions

    def replace(self, **kw):
        return dataclasses.replace(self, **kw)

    def gemm_flops(self):
        """Algorithmic GEMM flops (2*M*N*K) of forward, backward-data and weight-gradient passes."""
        G, H, T, B = self.G, self.hidden, self.T, self.B
        fwd = sum(2.0 * self.directions * T * B * G * H * (self.in_size(l) + H) for l in range(self.layers))
        return {"fwd": fwd, "bwd_data": fwd, "bwd_weights": fwd}


# The benchmark workloads (index 0 .. 4), a cell-variant workload (5) and a bidirectional stack (6).
WORKLOADS = [
    Workload("lstm_fp32_L1_T8_B4_H32", CELL_LSTM, 1, 8, 4, 32, 32, MODE_FP32,
             x_dist="uniform", forget_bias=1.0),
    Workload("lstm_bf16_L4_T100_B64_H512", CELL_LSTM, 4, 100, 64, 512, 512, MODE_BF16,
             forget_bias=1.0, state_std=0.1),
    Workload("lstm_bf16_L1_T1000_B4_H1024_infer", CELL_LSTM, 1, 1000, 4, 1024, 1024, MODE_BF16,
             forget_bias=1.0, training=False),
    Workload("lstm_bf16_L4_T50_B256_H4096", CELL_LSTM, 4, 50, 256, 4096, 4096, MODE_BF16,
             forget_bias=1.0),
    Workload("gru_bf16_L8_T200_B32_H1024", CELL_GRU, 8, 200, 32, 1024, 1024, MODE_BF16),
    # cell variant beyond the five: a 4-layer ReLU simple RNN, wide enough for the transposed steps
    Workload("relu_bf16_L4_T100_B256_H2048", CELL_RELU, 4, 100, 256, 2048, 2048, MODE_BF16),
    # bidirectional stack (beyond the five): 2 layers x 2 directions of a bf16 LSTM
    Workload("lstm_bf16_L2_T100_B128_H2048_bidir", CELL_LSTM, 2, 100, 128, 2048, 2048, MODE_BF16,
             forget_bias=1.0, directions=2),
]


def layer_weights(wl: Workload, l: int, dtype=np.float64, d: int = 0):
    """User-layout weights of direction ``d`` of layer ``l``:
    (W_x[G*H][I_l], W_h[G*H][H], b_x[G*H], b_h[G*H]).

    W_x and W_h ~ U(-1/sqrt(H), 1/sqrt(H)); biases are zero except the LSTM
    forget gate (gate block 1 of b_x), which gets ``forget_bias``.
    """
    G, H, I = wl.G, wl.hidden, wl.in_size(l)
    a = (0.05 if wl.kink_margin else 1.0) / math.sqrt(H)
    wx = uniform(wl.seed, 100 + 10 * l + 2 * d, (G * H, I), -a, a).astype(dtype)
    wh = uniform(wl.seed, 100 + 10 * l + 2 * d + 1, (G * H, H), -a, a).astype(dtype)
    bx = np.zeros(G * H, dtype=dtype)
    bh = np.zeros(G * H, dtype=dtype)
    if wl.cell == CELL_LSTM and wl.forget_bias:
        bx[H:2 * H] = wl.forget_bias
    if wl.kink_margin:
        bx[0::2] = wl.kink_margin
        bx[1::2] = -wl.kink_margin
    return wx, wh, bx, bh


def flat_weights(wl: Workload, dtype=np.float64) -> np.ndarray:
    """All layers' user-layout weights concatenated: per (layer, direction) W_x, W_h, b_x, b_h."""
    parts = []
    for l in range(wl.layers):
        for d in range(wl.directions):
            parts.extend(p.ravel() for p in layer_weights(wl, l, dtype, d))
    return np.concatenate(parts)


def make_x(wl: Workload, T=None, dtype=np.float64):
    T = wl.T if T is None else T
    shape = (T, wl.B, wl.input)
    if wl.x_dist == "uniform":
        return uniform(wl.seed, TID_X, shape, -1.0, 1.0).astype(dtype)
    return normal(wl.seed, TID_X, shape).astype(dtype)


def make_state(wl: Workload, which: str, dtype=np.float64):
    """h0 or c0, shape [L*D][B][H]."""
    shape = (wl.states, wl.B, wl.hidden)
    if wl.state_std == 0.0:
        return np.zeros(shape, dtype=dtype)
    tid = TID_H0 if which == "h0" else TID_C0
    return normal(wl.seed, tid, shape, std=wl.state_std).astype(dtype)


def make_dy(wl: Workload, T=None, dtype=np.float64):
    T = wl.T if T is None else T
    return normal(wl.seed, TID_DY, (T, wl.B, wl.directions * wl.hidden)).astype(dtype)


def make_dstate(wl: Workload, which: str, dtype=np.float64):
    """dhT or dcT [L*D][B][H] ~ N(0,1); the benchmark workloads pass none (zero)."""
    tid = TID_DHT if which == "dhT" else TID_DCT
    return normal(wl.seed, tid, (wl.states, wl.B, wl.hidden)).astype(dtype)


def round_bf16(a) -> np.ndarray:
    """Round to the nearest bfloat16 (via float32, ties to even), returned as float64."""
    t = torch.as_tensor(np.asarray(a)).to(torch.float32).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


def device_tensor(wl: Workload, what: str, device, dtype):
    """Draw one input directly on `device` (same counters as the host arrays;
    transcendental rounding of the normal transform may differ in the last
    ulp).  what: "x", "dy", "h0", "c0", "w"."""
    if what == "x":
        shape = (wl.T, wl.B, wl.input)
        if wl.x_dist == "uniform":
            t = uniform_t(wl.seed, TID_X, shape, -1.0, 1.0, device)
        else:
            t = normal_t(wl.seed, TID_X, shape, device=device)
    elif what == "dy":
        t = normal_t(wl.seed, TID_DY, (wl.T, wl.B, wl.directions * wl.hidden), device=device)
    elif what in ("h0", "c0"):
        shape = (wl.states, wl.B, wl.hidden)
        if wl.state_std == 0.0:
            t = torch.zeros(shape, dtype=torch.float64, device=device)
        else:
            t = normal_t(wl.seed, TID_H0 if what == "h0" else TID_C0, shape, std=wl.state_std, device=device)
    elif what == "w":
        parts = []
        for l, d in ((l, d) for l in range(wl.layers) for d in range(wl.directions)):
            G, H, I = wl.G, wl.hidden, wl.in_size(l)
            a = (0.05 if wl.kink_margin else 1.0) / math.sqrt(H)
            parts.append(uniform_t(wl.seed, 100 + 10 * l + 2 * d, (G * H * I,), -a, a, device).to(torch.float32))
            parts.append(uniform_t(wl.seed, 100 + 10 * l + 2 * d + 1, (G * H * H,), -a, a, device).to(torch.float32))
            bx = torch.zeros(G * H, dtype=torch.float32, device=device)
            if wl.cell == CELL_LSTM and wl.forget_bias:
                bx[H:2 * H] = wl.forget_bias
            if wl.kink_margin:
                bx[0::2] = wl.kink_margin
                bx[1::2] = -wl.kink_margin
            parts.append(bx)
            parts.append(torch.zeros(G * H, dtype=torch.float32, device=device))
        t = torch.cat(parts)
    else:
        raise ValueError(what)
    return t.to(torch.float32).to(dtype)
