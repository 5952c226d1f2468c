"""Double-precision CPU oracle for stacked LSTM / GRU / tanh-RNN (fwd + BPTT + dW).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg may import this package.  The
product library never loads it and shares no code with it.

The arithmetic lives in ``rnn_ref.cpp`` (plain C++17 loops in double,
OpenMP over batch rows / gate rows).  This module compiles it with the host
compiler and wraps its two entry points with ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rnn_ref.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "librnn_ref.so")
_lib = None

GATES = {0: 4, 1: 3, 2: 1, 3: 1}


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/librnn_ref.so (host compiler, -O2, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB) or
             os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC),
                                          os.path.getmtime(os.path.join(_HERE, "rnn_ref.h"))))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-std=c++17", "-O2", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        dp = ctypes.POINTER(ctypes.c_double)
        ci = ctypes.c_int
        lib.rnn_ref_fwd.argtypes = [ci] * 6 + [dp] * 7
        lib.rnn_ref_fwd.restype = ci
        lib.rnn_ref_bwd.argtypes = [ci] * 6 + [dp] * 11
        lib.rnn_ref_bwd.restype = ci
        ip = ctypes.POINTER(ctypes.c_int)
        lib.rnn_ref_fwd_len.argtypes = [ci] * 6 + [ip] + [dp] * 7
        lib.rnn_ref_fwd_len.restype = ci
        lib.rnn_ref_bwd_len.argtypes = [ci] * 6 + [ip] + [dp] * 11
        lib.rnn_ref_bwd_len.restype = ci
        lib.rnn_ref_fwd_dir.argtypes = [ci] * 7 + [ip] + [dp] * 7
        lib.rnn_ref_fwd_dir.restype = ci
        lib.rnn_ref_bwd_dir.argtypes = [ci] * 7 + [ip] + [dp] * 11
        lib.rnn_ref_bwd_dir.restype = ci
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.rnn_ref_fwd_kp.argtypes = [ci] * 7 + [ip, ci, u8p, dp] + [dp] * 7
        lib.rnn_ref_fwd_kp.restype = ci
        lib.rnn_ref_bwd_kp.argtypes = [ci] * 7 + [ip, ci, u8p] + [dp] * 11
        lib.rnn_ref_bwd_kp.restype = ci
        lib.rnn_ref_threads.restype = ci
        _lib = lib
    return _lib


def threads() -> int:
    return int(_load().rnn_ref_threads())


def _p(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _c(a, shape=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.float64)
    if shape is not None:
        assert a.shape == tuple(shape), (a.shape, shape)
    return a


def weight_count(cell, L, I, H, D=1):
    """Length of the flat weight vector: per (layer, direction) W_x, W_h, b_x, b_h."""
    G = GATES[cell]
    return sum(D * (G * H * ((I if l == 0 else D * H) + H) + 2 * G * H) for l in range(L))


def _lens(lens, T, B):
    if lens is None:
        return None
    a = np.ascontiguousarray(lens, dtype=np.int32)
    assert a.shape == (B,)
    return a


def _ip(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def _on(on, cell, L, T, B, H, D, decide):
    """uint8 decisions array [L*D][T][B][H]: given (decide = 3) or to be filled."""
    if cell != 3:
        return None
    if decide == 3:
        if on is None:
            raise ValueError("decide=3 needs the decisions `on`")
        a = np.ascontiguousarray(on, dtype=np.uint8)
        assert a.shape == (L * D, T, B, H)
        return a
    return np.zeros((L * D, T, B, H), np.uint8)


def _u8(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def relu_decisions(L, T, B, I, H, x, w, h0=None, lens=None, D=1, decide=1):
    """ReLU cell: (decisions uint8 [L*D][T][B][H], pre-activations [L*D][T][B][H])
    of the forward pass that takes the decisions in precision `decide`."""
    lens = _lens(lens, T, B)
    x = _c(x, (T, B, I))
    w = _c(w, (weight_count(3, L, I, H, D),))
    h0 = _c(h0, (L * D, B, H))
    on = np.zeros((L * D, T, B, H), np.uint8)
    pre = np.zeros((L * D, T, B, H))
    y = np.zeros((T, B, D * H))
    hT = np.zeros((L * D, B, H))
    rc = _load().rnn_ref_fwd_kp(3, L, D, T, B, I, H, _ip(lens), int(decide), _u8(on), _p(pre), _p(x), _p(h0), None,
                                _p(w), _p(y), _p(hT), None)
    if rc != 0:
        raise ValueError(f"rnn_ref_fwd_kp rejected its arguments ({rc})")
    return on, pre


def fwd(cell, L, T, B, I, H, x, w, h0=None, c0=None, lens=None, D=1, decide=0, on=None):
    """Forward pass. Returns (y[T][B][D*H], hT[L*D][B][H], cT[L*D][B][H] or None).
    lens[B] (optional): per-sequence lengths; later outputs are 0 and hT / cT
    are each sequence's state after its own last step.  D = 2: bidirectional
    layers (direction 1 runs time backwards; states indexed layer * 2 + direction).
    decide (ReLU cell): 0 decides on/off in double, 1 / 2 as a device storing
    h in bf16 / fp32 would, 3 takes the decisions `on` [L*D][T][B][H]
    (values stay double, see rnn_ref.h)."""
    lens = _lens(lens, T, B)
    x = _c(x, (T, B, I))
    w = _c(w, (weight_count(cell, L, I, H, D),))
    h0 = _c(h0, (L * D, B, H))
    c0 = _c(c0, (L * D, B, H)) if cell == 0 else None
    y = np.zeros((T, B, D * H))
    hT = np.zeros((L * D, B, H))
    cT = np.zeros((L * D, B, H)) if cell == 0 else None
    onb = _on(on, cell, L, T, B, H, D, decide)
    rc = _load().rnn_ref_fwd_kp(cell, L, D, T, B, I, H, _ip(lens), int(decide), _u8(onb), None, _p(x), _p(h0),
                                _p(c0), _p(w), _p(y), _p(hT), _p(cT))
    if rc != 0:
        raise ValueError(f"rnn_ref_fwd rejected its arguments ({rc})")
    return y, hT, cT


def bwd(cell, L, T, B, I, H, x, w, dy, h0=None, c0=None, dhT=None, dcT=None, lens=None, D=1, decide=0, on=None):
    """Backward pass. Returns (dx[T][B][I], dh0[L*D][B][H], dc0 or None, dw like w).
    decide: as for fwd."""
    lens = _lens(lens, T, B)
    x = _c(x, (T, B, I))
    w = _c(w, (weight_count(cell, L, I, H, D),))
    dy = _c(dy, (T, B, D * H))
    h0 = _c(h0, (L * D, B, H))
    c0 = _c(c0, (L * D, B, H)) if cell == 0 else None
    dhT = _c(dhT, (L * D, B, H))
    dcT = _c(dcT, (L * D, B, H)) if cell == 0 else None
    dx = np.zeros((T, B, I))
    dh0 = np.zeros((L * D, B, H))
    dc0 = np.zeros((L * D, B, H)) if cell == 0 else None
    dw = np.zeros_like(w)
    onb = _on(on, cell, L, T, B, H, D, decide)
    rc = _load().rnn_ref_bwd_kp(cell, L, D, T, B, I, H, _ip(lens), int(decide), _u8(onb), _p(x), _p(h0), _p(c0),
                                _p(w), _p(dy), _p(dhT), _p(dcT), _p(dx), _p(dh0), _p(dc0), _p(dw))
    if rc != 0:
        raise ValueError(f"rnn_ref_bwd rejected its arguments ({rc})")
    return dx, dh0, dc0, dw


def split_weights(cell, L, I, H, w, D=1):
    """Views (W_x, W_h, b_x, b_h) per (layer, direction) l * D + d of a flat
    user-layout weight vector."""
    G = GATES[cell]
    out, o = [], 0
    for l in range(L):
        for _ in range(D):
            In = I if l == 0 else D * H
            wx = w[o:o + G * H * In].reshape(G * H, In); o += G * H * In
            wh = w[o:o + G * H * H].reshape(G * H, H); o += G * H * H
            bx = w[o:o + G * H]; o += G * H
            bh = w[o:o + G * H]; o += G * H
            out.append((wx, wh, bx, bh))
    return out
