"""Caller-side plumbing: allocate the buffers librnn asks for with PyTorch,
upload seeded synthetic inputs, and drive forward / backward / weight-gradient
calls through the C-ABI binding.  No arithmetic of the method happens here.
"""
from __future__ import annotations

import numpy as np
import torch

from . import rnn, synth


def storage_dtype(mode):
    return torch.bfloat16 if mode == synth.MODE_BF16 else torch.float32


def as_storage(a: np.ndarray, mode) -> np.ndarray:
    """The values the device will hold for a storage-type tensor (bf16-rounded in bf16 mode)."""
    return synth.round_bf16(a) if mode == synth.MODE_BF16 else np.asarray(a, np.float32).astype(np.float64)


def as_f32(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, np.float32).astype(np.float64)


class HostInputs:
    """Synthetic inputs of a workload as float64 arrays holding exactly the
    values the device receives (storage-type rounding applied)."""

    def __init__(self, wl: synth.Workload, with_state_grads=False):
        m = wl.mode
        self.wl = wl
        self.x = as_storage(synth.make_x(wl), m)
        self.w = np.concatenate([as_storage(synth.layer_weights(wl, l, d=d)[k].ravel(), m)
                                 for l in range(wl.layers) for d in range(wl.directions) for k in range(4)])
        self.h0 = as_storage(synth.make_state(wl, "h0"), m)
        self.c0 = as_f32(synth.make_state(wl, "c0")) if wl.cell == synth.CELL_LSTM else None
        self.dy = as_storage(synth.make_dy(wl), m)
        self.dhT = as_storage(synth.make_dstate(wl, "dhT"), m) if with_state_grads else None
        self.dcT = (as_f32(synth.make_dstate(wl, "dcT"))
                    if with_state_grads and wl.cell == synth.CELL_LSTM else None)

    def columns(self, cols):
        """A copy restricted to batch columns `cols` (sequences are independent)."""
        out = object.__new__(HostInputs)
        out.wl = self.wl.replace(B=len(cols))
        out.w = self.w
        out.x = self.x[:, cols]
        out.h0 = self.h0[:, cols]
        out.c0 = None if self.c0 is None else self.c0[:, cols]
        out.dy = self.dy[:, cols]
        out.dhT = None if self.dhT is None else self.dhT[:, cols]
        out.dcT = None if self.dcT is None else self.dcT[:, cols]
        return out


def _dev(a, dtype, device):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device=device, dtype=dtype)


class Runner:
    """Device buffers + a librnn handle for one workload."""

    def __init__(self, wl: synth.Workload, device="cuda", flags=0, chunk=0, timeout_ns=0):
        self.wl = wl
        self.device = torch.device(device)
        self.r = rnn.RNN.for_workload(wl, flags=flags, chunk=chunk, timeout_ns=timeout_ns)
        self.sz = self.r.sizes()
        self.dt = storage_dtype(wl.mode)
        u8 = dict(dtype=torch.uint8, device=self.device)
        self.w_packed = torch.empty(self.sz["packed_weights"], **u8)
        self.ws = torch.zeros(self.sz["workspace"], **u8)
        self.reserve = torch.empty(self.sz["reserve"], **u8) if wl.training else None
        L, T, B, I, H = wl.layers, wl.T, wl.B, wl.input, wl.hidden
        f = dict(dtype=self.dt, device=self.device)
        S, D = wl.states, wl.directions
        self.y = torch.empty(T, B, D * H, **f)
        self.hT = torch.empty(S, B, H, **f)
        self.cT = torch.empty(S, B, H, dtype=torch.float32, device=self.device) if wl.cell == 0 else None
        if wl.training:
            self.dx = torch.empty(T, B, I, **f)
            self.dh0 = torch.empty(S, B, H, **f)
            self.dc0 = torch.empty(S, B, H, dtype=torch.float32, device=self.device) if wl.cell == 0 else None
            self.dw = torch.empty(self.sz["user_weights"] // (2 if wl.mode == 1 else 4), dtype=torch.float32,
                                  device=self.device)
        self.x = self.h0 = self.c0 = self.dy = self.dhT = self.dcT = self.w_user = None

    def upload(self, hi: HostInputs, state=True):
        d = self.device
        self.x = _dev(hi.x, self.dt, d)
        self.w_user = _dev(hi.w, self.dt, d)
        self.h0 = _dev(hi.h0, self.dt, d) if state else None
        self.c0 = _dev(hi.c0, torch.float32, d) if state else None
        self.dy = _dev(hi.dy, self.dt, d)
        self.dhT = _dev(hi.dhT, self.dt, d)
        self.dcT = _dev(hi.dcT, torch.float32, d)
        self.pack()

    def pack(self):
        self.r.pack_weights(self.w_user, self.w_packed)

    def forward(self, train=None):
        train = self.wl.training if train is None else train
        self.r.fwd(self.x, self.w_packed, self.y, self.ws, h0=self.h0, c0=self.c0, hT=self.hT, cT=self.cT,
                   reserve=self.reserve if train else None)

    def backward(self):
        self.r.bwd_data(self.dy, self.w_packed, self.reserve, self.ws, dhT=self.dhT, dcT=self.dcT, h0=self.h0,
                        c0=self.c0, dx=self.dx, dh0=self.dh0, dc0=self.dc0)

    def weights(self, accumulate=False):
        self.r.bwd_weights(self.x, self.reserve, self.dw, self.ws, h0=self.h0, accumulate=accumulate)

    def step(self):
        """One training step (forward, BPTT, weight gradients) or one inference forward."""
        if self.wl.training:
            self.forward(True)
            self.backward()
            self.weights()
        else:
            self.forward(False)

    def status(self):
        return self.r.sync_status(self.ws)

    def outputs(self):
        def h(t):
            return None if t is None else t.float().cpu().numpy().astype(np.float64)
        out = dict(y=h(self.y), hT=h(self.hT), cT=h(self.cT))
        if self.wl.training:
            out.update(dx=h(self.dx), dh0=h(self.dh0), dc0=h(self.dc0), dw=h(self.dw))
        return out
