"""Writes the oracle regression fixtures in this folder.

Every stored value comes from ``oracle`` alone (the double-precision CPU
definition of the LSTM / GRU / tanh- and ReLU-RNN cells, also bidirectional
and with per-sequence lengths, written out because the pages
of "Optimizing Performance of Recurrent Neural Networks on GPUs" name the
cells in their section "제안 방법" but print no equations).  Inputs are the
seeded synthetic generator's, so the fixture can be rebuilt byte for byte:

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from recurrent_neural_network_gb300 import synth  # noqa: E402

CASES = [
    # name, cell, L, T, B, I, H, directions, lengths
    ("lstm_L2_T3_B2_I3_H4", 0, 2, 3, 2, 3, 4, 1, None),
    ("gru_L2_T3_B2_I3_H4", 1, 2, 3, 2, 3, 4, 1, None),
    ("tanh_L2_T3_B2_I3_H4", 2, 2, 3, 2, 3, 4, 1, None),
    ("relu_L2_T3_B2_I3_H4", 3, 2, 3, 2, 3, 4, 1, None),
    ("lstm_bidir_L2_T3_B2_I3_H4", 0, 2, 3, 2, 3, 4, 2, None),
    ("gru_bidir_len_L2_T4_B3_I3_H4", 1, 2, 4, 3, 3, 4, 2, [4, 2, 1]),
]


def inputs(cell, L, T, B, I, H, D=1):
    wl = synth.Workload("golden", cell, L, T, B, I, H, synth.MODE_FP32, forget_bias=1.0, state_std=0.5,
                        directions=D)
    w = synth.flat_weights(wl)
    x = synth.make_x(wl)
    h0 = synth.make_state(wl, "h0")
    c0 = synth.make_state(wl, "c0")
    dy = synth.make_dy(wl)
    dhT = synth.make_dstate(wl, "dhT")
    dcT = synth.make_dstate(wl, "dcT")
    return w, x, h0, c0, dy, dhT, dcT


def compute(cell, L, T, B, I, H, D=1, lens=None):
    w, x, h0, c0, dy, dhT, dcT = inputs(cell, L, T, B, I, H, D)
    y, hT, cT = oracle.fwd(cell, L, T, B, I, H, x, w, h0=h0, c0=c0, lens=lens, D=D)
    dx, dh0, dc0, dw = oracle.bwd(cell, L, T, B, I, H, x, w, dy, h0=h0, c0=c0, dhT=dhT, dcT=dcT, lens=lens, D=D)
    out = dict(y=y, hT=hT, dx=dx, dh0=dh0, dw=dw)
    if cell == 0:
        out.update(cT=cT, dc0=dc0)
    return {k: [float(v) for v in np.asarray(a).ravel()] for k, a in out.items()}


def main():
    for name, *shape in CASES:
        rec = dict(case=name, shape=dict(zip(["cell", "L", "T", "B", "I", "H", "D", "lens"], shape)),
                   source="oracle (double precision), seeded synthetic inputs, seed 0",
                   values=compute(*shape))
        with open(os.path.join(HERE, name + ".json"), "w") as f:
            json.dump(rec, f, indent=0)


if __name__ == "__main__":
    main()
