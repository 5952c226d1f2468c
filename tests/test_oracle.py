"""Pins of the double-precision oracle to things other than itself.

Each test checks the oracle against the mathematics the cells are defined by
(closed forms, invariants, central finite differences), against a library
routine that implements the same textbook cells (PyTorch CPU float64
nn.LSTM / nn.GRU / nn.RNN with autograd), or against structural properties
(layer chaining, batch independence, T=1 reduction).  Together they fail on a
dropped term, a wrong sign, a wrong index or a transposed operand anywhere in
the forward pass, the BPTT recursion or the weight gradients.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from recurrent_neural_network_gb300 import synth

CELLS = [0, 1, 2, 3]
G = {0: 4, 1: 3, 2: 1, 3: 1}


def rand_case(cell, L, T, B, I, H, seed):
    rng = np.random.default_rng(seed)
    n = oracle.weight_count(cell, L, I, H)
    w = rng.uniform(-0.6, 0.6, n)
    x = rng.normal(size=(T, B, I))
    h0 = rng.normal(scale=0.5, size=(L, B, H))
    c0 = rng.normal(scale=0.5, size=(L, B, H))
    dy = rng.normal(size=(T, B, H))
    dhT = rng.normal(size=(L, B, H))
    dcT = rng.normal(size=(L, B, H))
    return w, x, h0, c0, dy, dhT, dcT


def torch_model(cell, L, I, H, w):
    if cell == 0:
        m = torch.nn.LSTM(I, H, L, dtype=torch.float64)
    elif cell == 1:
        m = torch.nn.GRU(I, H, L, dtype=torch.float64)
    else:
        m = torch.nn.RNN(I, H, L, nonlinearity="tanh" if cell == 2 else "relu", dtype=torch.float64)
    for l, (wx, wh, bx, bh) in enumerate(oracle.split_weights(cell, L, I, H, w)):
        getattr(m, f"weight_ih_l{l}").data.copy_(torch.from_numpy(wx))
        getattr(m, f"weight_hh_l{l}").data.copy_(torch.from_numpy(wh))
        getattr(m, f"bias_ih_l{l}").data.copy_(torch.from_numpy(bx))
        getattr(m, f"bias_hh_l{l}").data.copy_(torch.from_numpy(bh))
    return m


def torch_run(cell, L, T, B, I, H, w, x, h0, c0, dy, dhT, dcT):
    m = torch_model(cell, L, I, H, w)
    xt = torch.tensor(x, requires_grad=True)
    h0t = torch.tensor(h0, requires_grad=True)
    c0t = torch.tensor(c0, requires_grad=True)
    if cell == 0:
        y, (hT, cT) = m(xt, (h0t, c0t))
        loss = (y * torch.tensor(dy)).sum() + (hT * torch.tensor(dhT)).sum() + (cT * torch.tensor(dcT)).sum()
    else:
        y, hT = m(xt, h0t)
        cT = None
        loss = (y * torch.tensor(dy)).sum() + (hT * torch.tensor(dhT)).sum()
    loss.backward()
    dw = []
    for l in range(L):
        for nm in ("weight_ih", "weight_hh", "bias_ih", "bias_hh"):
            dw.append(getattr(m, f"{nm}_l{l}").grad.numpy().ravel())
    return dict(y=y.detach().numpy(), hT=hT.detach().numpy(),
                cT=None if cT is None else cT.detach().numpy(),
                dx=xt.grad.numpy(), dh0=h0t.grad.numpy(),
                dc0=c0t.grad.numpy() if cell == 0 else None, dw=np.concatenate(dw))


def oracle_run(cell, L, T, B, I, H, w, x, h0, c0, dy, dhT, dcT):
    y, hT, cT = oracle.fwd(cell, L, T, B, I, H, x, w, h0=h0, c0=c0)
    dx, dh0, dc0, dw = oracle.bwd(cell, L, T, B, I, H, x, w, dy, h0=h0, c0=c0, dhT=dhT, dcT=dcT)
    return dict(y=y, hT=hT, cT=cT, dx=dx, dh0=dh0, dc0=dc0, dw=dw)


# ---------------------------------------------------------------- library routine

@pytest.mark.parametrize("cell", CELLS)
@pytest.mark.parametrize("shape", [(2, 3, 2, 3, 2), (1, 8, 4, 32, 32), (3, 5, 3, 7, 6)])
def test_matches_torch_float64(cell, shape):
    L, T, B, I, H = shape
    args = rand_case(cell, L, T, B, I, H, seed=11 + cell)
    o = oracle_run(cell, L, T, B, I, H, *args)
    r = torch_run(cell, L, T, B, I, H, *args)
    for k in o:
        if o[k] is None:
            continue
        np.testing.assert_allclose(o[k], r[k], rtol=1e-10, atol=1e-12, err_msg=k)


def test_matches_torch_on_tiny_fp32_workload():
    wl = synth.WORKLOADS[0]
    w = synth.flat_weights(wl)
    x = synth.make_x(wl)
    z = np.zeros((wl.layers, wl.B, wl.hidden))
    dy = synth.make_dy(wl)
    args = (w, x, z, z, dy, z, z)
    o = oracle_run(0, wl.layers, wl.T, wl.B, wl.input, wl.hidden, *args)
    r = torch_run(0, wl.layers, wl.T, wl.B, wl.input, wl.hidden, *args)
    for k in o:
        np.testing.assert_allclose(o[k], r[k], rtol=1e-10, atol=1e-12, err_msg=k)


# ---------------------------------------------------------------- closed forms

def sig(a):
    return 1.0 / (1.0 + math.exp(-a))


def test_lstm_closed_form_zero_weights():
    """W = 0 makes the gates constant: c_t = f^(t+1) c0 + i g (1 - f^(t+1)) / (1 - f), h_t = o tanh(c_t)."""
    L, T, B, I, H = 1, 7, 2, 3, 2
    n = oracle.weight_count(0, L, I, H)
    w = np.zeros(n)
    _, _, bx, bh = oracle.split_weights(0, L, I, H, w)[0]
    bi, bf, bg, bo = 0.3, 1.0, -0.7, 0.2
    bx[0:H], bx[H:2 * H], bx[2 * H:3 * H], bx[3 * H:] = bi, bf, bg, bo
    bh[:] = 0.05
    x = np.random.default_rng(0).normal(size=(T, B, I))
    c0 = np.full((L, B, H), 0.4)
    y, hT, cT = oracle.fwd(0, L, T, B, I, H, x, w, c0=c0)
    i, f, g, o = sig(bi + .05), sig(bf + .05), math.tanh(bg + .05), sig(bo + .05)
    for t in range(T):
        c = f ** (t + 1) * 0.4 + i * g * (1 - f ** (t + 1)) / (1 - f)
        np.testing.assert_allclose(y[t], o * math.tanh(c), rtol=1e-13)
    np.testing.assert_allclose(cT, f ** T * 0.4 + i * g * (1 - f ** T) / (1 - f), rtol=1e-13)


def test_gru_closed_form_zero_weights():
    """W = 0: n = tanh(b_xn + r b_hn) is constant, h_t = z^(t+1) h0 + (1 - z^(t+1)) n."""
    L, T, B, I, H = 1, 6, 3, 2, 4
    w = np.zeros(oracle.weight_count(1, L, I, H))
    _, _, bx, bh = oracle.split_weights(1, L, I, H, w)[0]
    bx[:H], bx[H:2 * H], bx[2 * H:] = -0.2, 0.6, 0.35
    bh[:H], bh[H:2 * H], bh[2 * H:] = 0.1, -0.3, 0.8
    x = np.random.default_rng(1).normal(size=(T, B, I))
    h0 = np.full((L, B, H), -0.5)
    y, _, _ = oracle.fwd(1, L, T, B, I, H, x, w, h0=h0)
    r, z = sig(-0.1), sig(0.3)
    n = math.tanh(0.35 + r * 0.8)
    for t in range(T):
        np.testing.assert_allclose(y[t], z ** (t + 1) * -0.5 + (1 - z ** (t + 1)) * n, rtol=1e-13)


def test_rnn_closed_form_zero_weights():
    L, T, B, I, H = 2, 4, 2, 3, 5
    w = np.zeros(oracle.weight_count(2, L, I, H))
    for l, (_, _, bx, bh) in enumerate(oracle.split_weights(2, L, I, H, w)):
        bx[:] = 0.25 * (l + 1)
        bh[:] = -0.1
    x = np.random.default_rng(2).normal(size=(T, B, I))
    y, hT, _ = oracle.fwd(2, L, T, B, I, H, x, w, h0=np.ones((L, B, H)))
    np.testing.assert_allclose(y, math.tanh(0.5 - 0.1), rtol=1e-14)
    np.testing.assert_allclose(hT[0], math.tanh(0.25 - 0.1), rtol=1e-14)


def test_relu_rnn_closed_form_zero_weights():
    """Zero weights: every step of every layer is max(0, b_x + b_h) (0 where
    that sum is negative), whatever x and h0 are."""
    L, T, B, I, H = 2, 4, 2, 3, 4
    w = np.zeros(oracle.weight_count(3, L, I, H))
    for l, (_, _, bx, bh) in enumerate(oracle.split_weights(3, L, I, H, w)):
        bx[:] = [0.3, -0.2, 0.05 * (l + 1), -1.0]
        bh[:] = 0.1
    x = np.random.default_rng(4).normal(size=(T, B, I))
    y, hT, _ = oracle.fwd(3, L, T, B, I, H, x, w, h0=np.ones((L, B, H)))
    want = np.maximum(0.0, np.array([0.4, -0.1, 0.2, -0.9]))
    np.testing.assert_allclose(y, np.broadcast_to(want, y.shape), rtol=1e-14, atol=0)
    np.testing.assert_allclose(hT[0], np.broadcast_to(np.maximum(0.0, [0.4, -0.1, 0.15, -0.9]), hT[0].shape),
                               rtol=1e-14, atol=0)


def test_relu_rnn_gradient_is_masked_by_the_activation():
    """One step, one unit: dL/da = dy where a > 0 and exactly 0 where a < 0,
    so dx = dy * w_x on active entries and 0 elsewhere."""
    L, T, B, I, H = 1, 1, 2, 1, 1
    w = np.array([2.0, 0.0, -0.5, 0.0])  # W_x, W_h, b_x, b_h
    x = np.array([[[1.0], [-1.0]]])       # a = 2x - 0.5: 1.5 (active), -2.5 (inactive)
    dy = np.array([[[3.0], [7.0]]])
    y, _, _ = oracle.fwd(3, L, T, B, I, H, x, w)
    np.testing.assert_array_equal(y.reshape(-1), [1.5, 0.0])
    dx, dh0, _, dw = oracle.bwd(3, L, T, B, I, H, x, w, dy)
    np.testing.assert_array_equal(dx.reshape(-1), [6.0, 0.0])
    np.testing.assert_array_equal(dw, [3.0, 0.0, 3.0, 3.0])  # dW_x = 3*1, dW_h = 3*h0 = 0, db = 3


def test_lstm_t1_single_unit_by_hand():
    """One step of a 1x1 LSTM written out scalar by scalar."""
    # w layout: Wx[4][1], Wh[4][1], bx[4], bh[4]
    wx = np.array([0.5, -0.25, 0.75, 1.0])
    wh = np.array([0.1, 0.2, -0.3, 0.4])
    bx = np.array([0.0, 1.0, 0.1, -0.1])
    bh = np.array([0.05, 0.0, 0.0, 0.2])
    w = np.concatenate([wx, wh, bx, bh])
    x = np.array([[[0.8]]])
    h0, c0 = np.array([[[0.3]]]), np.array([[[-0.6]]])
    y, hT, cT = oracle.fwd(0, 1, 1, 1, 1, 1, x, w, h0=h0, c0=c0)
    a = wx * 0.8 + bx + wh * 0.3 + bh
    i, f, g, o = sig(a[0]), sig(a[1]), math.tanh(a[2]), sig(a[3])
    c = f * -0.6 + i * g
    assert abs(cT[0, 0, 0] - c) < 1e-15
    assert abs(y[0, 0, 0] - o * math.tanh(c)) < 1e-15
    # backward of L = y: dh = 1
    dx, dh0, dc0, dw = oracle.bwd(0, 1, 1, 1, 1, 1, x, w, np.ones((1, 1, 1)), h0=h0, c0=c0)
    tau = math.tanh(c)
    dc = o * (1 - tau * tau)
    dga = np.array([dc * g * i * (1 - i), dc * -0.6 * f * (1 - f), dc * i * (1 - g * g), tau * o * (1 - o)])
    np.testing.assert_allclose(dw[0:4], dga * 0.8, rtol=1e-13)
    np.testing.assert_allclose(dw[4:8], dga * 0.3, rtol=1e-13)
    np.testing.assert_allclose(dw[8:12], dga, rtol=1e-13)
    np.testing.assert_allclose(dw[12:16], dga, rtol=1e-13)
    assert abs(dx[0, 0, 0] - (dga * wx).sum()) < 1e-14
    assert abs(dh0[0, 0, 0] - (dga * wh).sum()) < 1e-14
    assert abs(dc0[0, 0, 0] - dc * f) < 1e-15


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("cell", CELLS)
def test_zero_input_zero_state_zero_bias_stays_zero(cell):
    L, T, B, I, H = 2, 5, 3, 4, 6
    rng = np.random.default_rng(3)
    w = rng.uniform(-1, 1, oracle.weight_count(cell, L, I, H))
    for (_, _, bx, bh) in oracle.split_weights(cell, L, I, H, w):
        bx[:] = 0
        bh[:] = 0
    x = np.zeros((T, B, I))
    y, hT, cT = oracle.fwd(cell, L, T, B, I, H, x, w)
    assert not y.any() and not hT.any()
    if cell == 0:
        assert not cT.any()
    dy = rng.normal(size=(T, B, H))
    dx, dh0, dc0, dw = oracle.bwd(cell, L, T, B, I, H, x, w, dy)
    for (dwx, dwh, dbx, dbh) in oracle.split_weights(cell, L, I, H, dw):
        assert not dwx.any() and not dwh.any()   # every product has a zero operand
        if cell == 3:
            assert not dbx.any()  # every pre-activation is exactly 0, where ReLU's slope is taken as 0
        else:
            assert dbx.any()      # the bias gradient does not vanish


# ---------------------------------------------------------------- finite differences

def loss_of(cell, L, T, B, I, H, w, x, h0, c0, dy, dhT, dcT):
    y, hT, cT = oracle.fwd(cell, L, T, B, I, H, x, w, h0=h0, c0=c0)
    s = (y * dy).sum() + (hT * dhT).sum()
    if cell == 0:
        s += (cT * dcT).sum()
    return s


@pytest.mark.parametrize("cell", CELLS)
def test_central_finite_differences(cell):
    L, T, B, I, H = 2, 3, 2, 3, 2
    w, x, h0, c0, dy, dhT, dcT = rand_case(cell, L, T, B, I, H, seed=5 + cell)
    dx, dh0, dc0, dw = oracle.bwd(cell, L, T, B, I, H, x, w, dy, h0=h0, c0=c0, dhT=dhT, dcT=dcT)
    eps = 1e-6
    targets = [("w", w, dw), ("x", x, dx), ("h0", h0, dh0)]
    if cell == 0:
        targets.append(("c0", c0, dc0))
    for name, arr, grad in targets:
        flat = arr.reshape(-1)
        num = np.zeros(flat.size)
        for k in range(flat.size):
            save = flat[k]
            flat[k] = save + eps
            lp = loss_of(cell, L, T, B, I, H, w, x, h0, c0, dy, dhT, dcT)
            flat[k] = save - eps
            lm = loss_of(cell, L, T, B, I, H, w, x, h0, c0, dy, dhT, dcT)
            flat[k] = save
            num[k] = (lp - lm) / (2 * eps)
        scale = max(np.abs(num).max(), 1e-3)
        err = np.abs(num - grad.reshape(-1)).max() / scale
        assert err < 1e-7, (name, err)


# ---------------------------------------------------------------- structure

@pytest.mark.parametrize("cell", CELLS)
def test_stack_equals_chained_single_layers(cell):
    L, T, B, I, H = 3, 4, 2, 5, 3
    w, x, h0, c0, *_ = rand_case(cell, L, T, B, I, H, seed=21)
    y, hT, cT = oracle.fwd(cell, L, T, B, I, H, x, w, h0=h0, c0=c0)
    inp = x
    for l, parts in enumerate(oracle.split_weights(cell, L, I, H, w)):
        wl = np.concatenate([p.ravel() for p in parts])
        In = I if l == 0 else H
        inp, hl, cl = oracle.fwd(cell, 1, T, B, In, H, inp, wl, h0=h0[l:l + 1], c0=c0[l:l + 1])
        np.testing.assert_allclose(hl[0], hT[l], rtol=0, atol=0)
        if cell == 0:
            np.testing.assert_allclose(cl[0], cT[l], rtol=0, atol=0)
    np.testing.assert_allclose(inp, y, rtol=0, atol=0)


@pytest.mark.parametrize("cell", CELLS)
def test_batch_columns_are_independent(cell):
    L, T, B, I, H = 2, 4, 5, 3, 4
    w, x, h0, c0, dy, dhT, dcT = rand_case(cell, L, T, B, I, H, seed=31)
    full = oracle.bwd(cell, L, T, B, I, H, x, w, dy, h0=h0, c0=c0, dhT=dhT, dcT=dcT)
    perm = np.array([3, 0, 4, 1, 2])
    yf, _, _ = oracle.fwd(cell, L, T, B, I, H, x, w, h0=h0, c0=c0)
    yp, _, _ = oracle.fwd(cell, L, T, B, I, H, x[:, perm], w, h0=h0[:, perm], c0=c0[:, perm])
    np.testing.assert_allclose(yp, yf[:, perm], rtol=0, atol=1e-15)
    # one column alone gives that column's data gradients; dW sums over columns
    dw_sum = np.zeros_like(w)
    for b in range(B):
        s = slice(b, b + 1)
        dx, dh0, dc0, dw = oracle.bwd(cell, L, T, 1, I, H, x[:, s], w, dy[:, s], h0=h0[:, s], c0=c0[:, s],
                                      dhT=dhT[:, s], dcT=dcT[:, s])
        np.testing.assert_allclose(dx, full[0][:, s], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(dh0, full[1][:, s], rtol=1e-12, atol=1e-14)
        dw_sum += dw
    np.testing.assert_allclose(dw_sum, full[3], rtol=1e-11, atol=1e-13)


def test_prefix_in_time():
    """The first T' outputs do not depend on later inputs (causality)."""
    cell, L, T, B, I, H = 0, 2, 6, 2, 3, 4
    w, x, h0, c0, *_ = rand_case(cell, L, T, B, I, H, seed=41)
    y, _, _ = oracle.fwd(cell, L, T, B, I, H, x, w, h0=h0, c0=c0)
    y3, _, _ = oracle.fwd(cell, L, 3, B, I, H, x[:3], w, h0=h0, c0=c0)
    np.testing.assert_array_equal(y3, y[:3])


def test_rejects_bad_arguments():
    lib = oracle._load()
    x = np.zeros(1)
    w = np.zeros(oracle.weight_count(0, 1, 1, 1))
    p = oracle._p
    assert lib.rnn_ref_fwd(7, 1, 1, 1, 1, 1, p(x), None, None, p(w), None, None, None) == -1
    assert lib.rnn_ref_fwd(0, 0, 1, 1, 1, 1, p(x), None, None, p(w), None, None, None) == -1
    assert lib.rnn_ref_fwd(0, 1, 1, 1, 1, 1, p(x), None, None, None, None, None, None) == -1


# ---------------------------------------------------------------- stored fixtures

@pytest.mark.parametrize("name", ["lstm_L2_T3_B2_I3_H4", "gru_L2_T3_B2_I3_H4", "tanh_L2_T3_B2_I3_H4",
                                  "relu_L2_T3_B2_I3_H4", "lstm_bidir_L2_T3_B2_I3_H4",
                                  "gru_bidir_len_L2_T4_B3_I3_H4"])
def test_oracle_matches_stored_fixture(name):
    """Regression pin: the fixtures were written by tests/golden/make_golden.py from the oracle."""
    import json
    import os
    import sys
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    sys.path.insert(0, here)
    import make_golden
    rec = json.load(open(os.path.join(here, name + ".json")))
    sh = rec["shape"]
    now = make_golden.compute(sh["cell"], sh["L"], sh["T"], sh["B"], sh["I"], sh["H"], sh.get("D", 1), sh.get("lens"))
    for k, v in rec["values"].items():
        np.testing.assert_allclose(now[k], v, rtol=1e-12, atol=1e-14, err_msg=k)


# ---------------------------------------------------------------- variable lengths

LENS_CASES = [(0, [3, 1, 4, 2]), (1, [4, 4, 2, 1]), (2, [1, 3, 2, 4]), (3, [2, 4, 1, 3])]


@pytest.mark.parametrize("cell,lens", LENS_CASES, ids=["lstm", "gru", "tanh", "relu"])
def test_variable_lengths_equal_separate_truncated_runs(cell, lens):
    """A batch of sequences of different lengths equals running each sequence
    alone for its own number of steps: outputs (zero past the end), final
    states, data gradients, and weight gradients summed over the sequences."""
    L, T, B, I, H = 2, 4, 4, 3, 5
    w, x, h0, c0, dy, dhT, dcT = rand_case(cell, L, T, B, I, H, seed=41 + cell)
    y, hT, cT = oracle.fwd(cell, L, T, B, I, H, x, w, h0=h0, c0=c0, lens=lens)
    dx, dh0, dc0, dw = oracle.bwd(cell, L, T, B, I, H, x, w, dy, h0=h0, c0=c0, dhT=dhT, dcT=dcT, lens=lens)
    dw_sum = np.zeros_like(dw)
    for b, n in enumerate(lens):
        s = slice(b, b + 1)
        cb = c0[:, s] if cell == 0 else None
        yb, hb, cTb = oracle.fwd(cell, L, n, 1, I, H, x[:n, s], w, h0=h0[:, s], c0=cb)
        np.testing.assert_allclose(y[:n, s], yb, rtol=1e-13, atol=1e-15)
        assert not y[n:, b].any()
        np.testing.assert_allclose(hT[:, s], hb, rtol=1e-13, atol=1e-15)
        if cell == 0:
            np.testing.assert_allclose(cT[:, s], cTb, rtol=1e-13, atol=1e-15)
        dxb, dh0b, dc0b, dwb = oracle.bwd(cell, L, n, 1, I, H, x[:n, s], w, dy[:n, s], h0=h0[:, s], c0=cb,
                                          dhT=dhT[:, s], dcT=dcT[:, s] if cell == 0 else None)
        np.testing.assert_allclose(dx[:n, s], dxb, rtol=1e-12, atol=1e-14)
        assert not dx[n:, b].any()
        np.testing.assert_allclose(dh0[:, s], dh0b, rtol=1e-12, atol=1e-14)
        if cell == 0:
            np.testing.assert_allclose(dc0[:, s], dc0b, rtol=1e-12, atol=1e-14)
        dw_sum += dwb
    np.testing.assert_allclose(dw, dw_sum, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("cell,lens", LENS_CASES, ids=["lstm", "gru", "tanh", "relu"])
def test_variable_lengths_match_torch_packed_sequences(cell, lens):
    """PyTorch float64 on a packed batch (pack_padded_sequence) with autograd."""
    L, T, B, I, H = 2, 4, 4, 3, 5
    w, x, h0, c0, dy, dhT, dcT = rand_case(cell, L, T, B, I, H, seed=51 + cell)
    y, hT, cT = oracle.fwd(cell, L, T, B, I, H, x, w, h0=h0, c0=c0, lens=lens)
    dx, dh0, dc0, dw = oracle.bwd(cell, L, T, B, I, H, x, w, dy, h0=h0, c0=c0, dhT=dhT, dcT=dcT, lens=lens)
    m = torch_model(cell, L, I, H, w)
    xt = torch.tensor(x, requires_grad=True)
    h0t = torch.tensor(h0, requires_grad=True)
    c0t = torch.tensor(c0, requires_grad=True)
    packed = torch.nn.utils.rnn.pack_padded_sequence(xt, torch.tensor(lens), enforce_sorted=False)
    if cell == 0:
        out, (hTt, cTt) = m(packed, (h0t, c0t))
    else:
        out, hTt = m(packed, h0t)
    yt, _ = torch.nn.utils.rnn.pad_packed_sequence(out, total_length=T)
    loss = (yt * torch.tensor(dy)).sum() + (hTt * torch.tensor(dhT)).sum()
    if cell == 0:
        loss = loss + (cTt * torch.tensor(dcT)).sum()
    loss.backward()
    np.testing.assert_allclose(y, yt.detach().numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(hT, hTt.detach().numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dh0, h0t.grad.numpy(), rtol=1e-10, atol=1e-12)
    if cell == 0:
        np.testing.assert_allclose(cT, cTt.detach().numpy(), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(dc0, c0t.grad.numpy(), rtol=1e-10, atol=1e-12)
    tw = []
    for l in range(L):
        for nm in ("weight_ih", "weight_hh", "bias_ih", "bias_hh"):
            tw.append(getattr(m, f"{nm}_l{l}").grad.numpy().ravel())
    np.testing.assert_allclose(dw, np.concatenate(tw), rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- bidirectional layers

def rand_case_bidir(cell, L, T, B, I, H, seed):
    rng = np.random.default_rng(seed)
    n = oracle.weight_count(cell, L, I, H, D=2)
    w = rng.uniform(-0.6, 0.6, n)
    x = rng.normal(size=(T, B, I))
    h0 = rng.normal(scale=0.5, size=(2 * L, B, H))
    c0 = rng.normal(scale=0.5, size=(2 * L, B, H))
    dy = rng.normal(size=(T, B, 2 * H))
    dhT = rng.normal(size=(2 * L, B, H))
    dcT = rng.normal(size=(2 * L, B, H))
    return w, x, h0, c0, dy, dhT, dcT


def torch_bidir(cell, L, I, H, w):
    kw = dict(bidirectional=True, dtype=torch.float64)
    if cell == 0:
        m = torch.nn.LSTM(I, H, L, **kw)
    elif cell == 1:
        m = torch.nn.GRU(I, H, L, **kw)
    else:
        m = torch.nn.RNN(I, H, L, nonlinearity="tanh" if cell == 2 else "relu", **kw)
    views = oracle.split_weights(cell, L, I, H, w, D=2)
    for l in range(L):
        for d, sfx in enumerate(("", "_reverse")):
            wx, wh, bx, bh = views[2 * l + d]
            getattr(m, f"weight_ih_l{l}{sfx}").data.copy_(torch.from_numpy(wx))
            getattr(m, f"weight_hh_l{l}{sfx}").data.copy_(torch.from_numpy(wh))
            getattr(m, f"bias_ih_l{l}{sfx}").data.copy_(torch.from_numpy(bx))
            getattr(m, f"bias_hh_l{l}{sfx}").data.copy_(torch.from_numpy(bh))
    return m


def torch_bidir_run(cell, L, T, B, I, H, w, x, h0, c0, dy, dhT, dcT, lens=None):
    m = torch_bidir(cell, L, I, H, w)
    xt = torch.tensor(x, requires_grad=True)
    h0t = torch.tensor(h0, requires_grad=True)
    c0t = torch.tensor(c0, requires_grad=True)
    inp = xt if lens is None else torch.nn.utils.rnn.pack_padded_sequence(xt, torch.tensor(lens), enforce_sorted=False)
    if cell == 0:
        out, (hT, cT) = m(inp, (h0t, c0t))
    else:
        out, hT = m(inp, h0t)
        cT = None
    y = out if lens is None else torch.nn.utils.rnn.pad_packed_sequence(out, total_length=T)[0]
    loss = (y * torch.tensor(dy)).sum() + (hT * torch.tensor(dhT)).sum()
    if cell == 0:
        loss = loss + (cT * torch.tensor(dcT)).sum()
    loss.backward()
    dw = []
    for l in range(L):
        for sfx in ("", "_reverse"):
            for nm in ("weight_ih", "weight_hh", "bias_ih", "bias_hh"):
                dw.append(getattr(m, f"{nm}_l{l}{sfx}").grad.numpy().ravel())
    return dict(y=y.detach().numpy(), hT=hT.detach().numpy(),
                cT=None if cT is None else cT.detach().numpy(),
                dx=xt.grad.numpy(), dh0=h0t.grad.numpy(),
                dc0=c0t.grad.numpy() if cell == 0 else None, dw=np.concatenate(dw))


def oracle_bidir_run(cell, L, T, B, I, H, w, x, h0, c0, dy, dhT, dcT, lens=None):
    y, hT, cT = oracle.fwd(cell, L, T, B, I, H, x, w, h0=h0, c0=c0, lens=lens, D=2)
    dx, dh0, dc0, dw = oracle.bwd(cell, L, T, B, I, H, x, w, dy, h0=h0, c0=c0, dhT=dhT, dcT=dcT, lens=lens, D=2)
    return dict(y=y, hT=hT, cT=cT, dx=dx, dh0=dh0, dc0=dc0, dw=dw)


@pytest.mark.parametrize("cell", CELLS)
@pytest.mark.parametrize("shape", [(2, 3, 2, 3, 2), (3, 5, 3, 7, 6)])
def test_bidirectional_matches_torch_float64(cell, shape):
    """PyTorch float64 bidirectional nn.LSTM / GRU / RNN with autograd: outputs
    [forward, reverse] per timestep, final states per (layer, direction), and
    every gradient."""
    L, T, B, I, H = shape
    args = rand_case_bidir(cell, L, T, B, I, H, seed=71 + cell)
    o = oracle_bidir_run(cell, L, T, B, I, H, *args)
    r = torch_bidir_run(cell, L, T, B, I, H, *args)
    for k in o:
        if o[k] is None:
            continue
        np.testing.assert_allclose(o[k], r[k], rtol=1e-10, atol=1e-12, err_msg=k)


@pytest.mark.parametrize("cell,lens", LENS_CASES, ids=["lstm", "gru", "tanh", "relu"])
def test_bidirectional_variable_lengths_match_torch_packed(cell, lens):
    """Packed bidirectional batch: the reverse direction of each sequence starts
    at its own last step."""
    L, T, B, I, H = 2, 4, 4, 3, 5
    args = rand_case_bidir(cell, L, T, B, I, H, seed=81 + cell)
    o = oracle_bidir_run(cell, L, T, B, I, H, *args, lens=lens)
    r = torch_bidir_run(cell, L, T, B, I, H, *args, lens=lens)
    for k in o:
        if o[k] is None:
            continue
        np.testing.assert_allclose(o[k], r[k], rtol=1e-10, atol=1e-12, err_msg=k)


@pytest.mark.parametrize("cell", CELLS)
def test_bidirectional_single_layer_is_two_unidirectional_runs(cell):
    """One bidirectional layer = the forward-direction weights run on x, and the
    reverse-direction weights run on x reversed in time with the output
    reversed back (both by the unidirectional oracle)."""
    T, B, I, H = 5, 3, 4, 6
    w, x, h0, c0, dy, dhT, dcT = rand_case_bidir(cell, 1, T, B, I, H, seed=91 + cell)
    y, hT, cT = oracle.fwd(cell, 1, T, B, I, H, x, w, h0=h0, c0=c0, D=2)
    n1 = oracle.weight_count(cell, 1, I, H)
    c0f = c0[0:1] if cell == 0 else None
    c0r = c0[1:2] if cell == 0 else None
    yf, hf, cf = oracle.fwd(cell, 1, T, B, I, H, x, w[:n1], h0=h0[0:1], c0=c0f)
    yr, hr, cr = oracle.fwd(cell, 1, T, B, I, H, x[::-1], w[n1:], h0=h0[1:2], c0=c0r)
    np.testing.assert_allclose(y[:, :, :H], yf, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(y[:, :, H:], yr[::-1], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(hT[0], hf[0], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(hT[1], hr[0], rtol=1e-13, atol=1e-15)
    dx, dh0, dc0, dw = oracle.bwd(cell, 1, T, B, I, H, x, w, dy, h0=h0, c0=c0, dhT=dhT, dcT=dcT, D=2)
    dxf, dh0f, dc0f, dwf = oracle.bwd(cell, 1, T, B, I, H, x, w[:n1], dy[:, :, :H], h0=h0[0:1], c0=c0f,
                                      dhT=dhT[0:1], dcT=dcT[0:1] if cell == 0 else None)
    dxr, dh0r, dc0r, dwr = oracle.bwd(cell, 1, T, B, I, H, x[::-1], w[n1:], dy[::-1, :, H:], h0=h0[1:2], c0=c0r,
                                      dhT=dhT[1:2], dcT=dcT[1:2] if cell == 0 else None)
    np.testing.assert_allclose(dx, dxf + dxr[::-1], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dh0, np.concatenate([dh0f, dh0r]), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dw, np.concatenate([dwf, dwr]), rtol=1e-12, atol=1e-14)
    if cell == 0:
        np.testing.assert_allclose(cT, np.concatenate([cf, cr]), rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(dc0, np.concatenate([dc0f, dc0r]), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("cell", CELLS)
def test_bidirectional_central_finite_differences(cell):
    L, T, B, I, H = 2, 3, 2, 3, 2
    w, x, h0, c0, dy, dhT, dcT = rand_case_bidir(cell, L, T, B, I, H, seed=101 + cell)
    dx, dh0, dc0, dw = oracle.bwd(cell, L, T, B, I, H, x, w, dy, h0=h0, c0=c0, dhT=dhT, dcT=dcT, D=2)

    def loss():
        y, hT, cT = oracle.fwd(cell, L, T, B, I, H, x, w, h0=h0, c0=c0, D=2)
        v = float((y * dy).sum() + (hT * dhT).sum())
        return v + (float((cT * dcT).sum()) if cell == 0 else 0.0)

    eps = 1e-6
    targets = [("w", w, dw), ("x", x, dx), ("h0", h0, dh0)]
    if cell == 0:
        targets.append(("c0", c0, dc0))
    for name, arr, grad in targets:
        flat = arr.reshape(-1)
        num = np.zeros(flat.size)
        for k in range(flat.size):
            save = flat[k]
            flat[k] = save + eps
            lp = loss()
            flat[k] = save - eps
            lm = loss()
            flat[k] = save
            num[k] = (lp - lm) / (2 * eps)
        scale = max(np.abs(num).max(), 1e-3)
        err = np.abs(num - grad.reshape(-1)).max() / scale
        assert err < 1e-7, (name, err)


# ---------------------------------------------------------------- ReLU decisions in the device's precision

def test_relu_decisions_in_storage_precision_by_hand():
    """One unit, two steps, x chosen so that h_1 = 1 + 2^-10 and the second
    pre-activation a_2 = h_1 - (1 + 2^-11) = +2^-11 is on in double, while a
    device storing h_1 in bf16 (spacing 2^-7 at 1, so h_1 -> 1) sees
    a_2 = -2^-11 and switches the unit off.  fp32 holds 1 + 2^-10 exactly.
    Values stay double: h_1 is 1 + 2^-10 in every mode."""
    w = np.array([1.0, 1.0, 0.0, 0.0])  # W_x, W_h, b_x, b_h of a 1x1 ReLU cell
    x = np.array([1.0 + 2.0 ** -10, -(1.0 + 2.0 ** -11)]).reshape(2, 1, 1)
    dy = np.array([0.5, 2.0]).reshape(2, 1, 1)
    for decide, h2 in ((0, 2.0 ** -11), (2, 2.0 ** -11), (1, 0.0)):
        y, hT, _ = oracle.fwd(3, 1, 2, 1, 1, 1, x, w, decide=decide)
        assert y[0, 0, 0] == 1.0 + 2.0 ** -10 and y[1, 0, 0] == h2, (decide, y.ravel())
        dx, dh0, _, dw = oracle.bwd(3, 1, 2, 1, 1, 1, x, w, dy, decide=decide)
        on2 = h2 > 0
        # dL/da_2 = dy_2 if on; dL/da_1 = dy_1 + W_h dL/da_2 (unit 1 is on)
        da2 = 2.0 if on2 else 0.0
        da1 = 0.5 + da2
        np.testing.assert_allclose(dx.ravel(), [da1, da2], rtol=0, atol=0)
        np.testing.assert_allclose(dw, [da1 * x[0, 0, 0] + da2 * x[1, 0, 0], da2 * y[0, 0, 0], da1 + da2, da1 + da2],
                                   rtol=1e-15)


@pytest.mark.parametrize("cell", CELLS)
def test_decisions_in_storage_precision_leave_clear_cases_unchanged(cell):
    """Away from the kink (margin-shaped ReLU inputs) and for the other cells the
    kernel-precision decisions are the double ones, so every output and
    gradient is bit-identical to the plain definition."""
    wl = synth.Workload("dec", cell, 2, 5, 3, 6, 8, synth.MODE_BF16, forget_bias=1.0, state_std=0.3,
                        kink_margin=0.75 if cell == 3 else 0.0)
    from recurrent_neural_network_gb300 import runner
    hi = runner.HostInputs(wl, with_state_grads=True)
    ref = oracle.bwd(cell, 2, 5, 3, 6, 8, hi.x, hi.w, hi.dy, h0=hi.h0, c0=hi.c0, dhT=hi.dhT, dcT=hi.dcT)
    for decide in (1, 2):
        got = oracle.bwd(cell, 2, 5, 3, 6, 8, hi.x, hi.w, hi.dy, h0=hi.h0, c0=hi.c0, dhT=hi.dhT, dcT=hi.dcT,
                         decide=decide)
        for a, b in zip(got, ref):
            if a is not None:
                np.testing.assert_array_equal(a, b)
    with pytest.raises(ValueError):
        oracle.fwd(cell, 1, 2, 1, 1, 1, np.zeros((2, 1, 1)), np.zeros(oracle.weight_count(cell, 1, 1, 1)), decide=4)


def test_relu_decisions_in_storage_precision_with_ordinary_weights():
    """With ordinary weights a few bf16 decisions differ from the double ones
    (units whose pre-activation lies within bf16 rounding of 0): the forward
    outputs stay close (the function is continuous) and only a small share of
    the decisions changes."""
    wl = synth.Workload("dec", 3, 1, 20, 6, 16, 64, synth.MODE_BF16, state_std=0.3)
    from recurrent_neural_network_gb300 import runner
    hi = runner.HostInputs(wl)
    y0, _, _ = oracle.fwd(3, 1, 20, 6, 16, 64, hi.x, hi.w, h0=hi.h0)
    y1, _, _ = oracle.fwd(3, 1, 20, 6, 16, 64, hi.x, hi.w, h0=hi.h0, decide=1)
    assert np.abs(y0 - y1).max() < 1e-2
    on0, on1 = y0 > 0, (y1 > 0) | (y1 < 0)  # imposed "on" may carry a pre-activation just below 0
    changed = int((on0 != on1).sum())
    assert 0 < changed < on0.size // 100, changed


def test_relu_given_decisions_reproduce_the_taken_ones():
    """Decisions taken in bf16 precision and handed back (decide = 3) give the
    same outputs and gradients bit for bit; the pre-activations returned are
    consistent with them (on exactly where the bf16-pass pre-activation > 0,
    and h = max(0, a) when decided in double)."""
    wl = synth.Workload("dec", 3, 2, 7, 4, 16, 32, synth.MODE_BF16, state_std=0.3)
    from recurrent_neural_network_gb300 import runner
    hi = runner.HostInputs(wl, with_state_grads=True)
    args = (3, 2, 7, 4, 16, 32, hi.x, hi.w)
    on, pre = oracle.relu_decisions(2, 7, 4, 16, 32, hi.x, hi.w, h0=hi.h0, decide=1)
    np.testing.assert_array_equal(on, (pre > 0).astype(np.uint8))
    a = oracle.bwd(*args, hi.dy, h0=hi.h0, dhT=hi.dhT, decide=1)
    b = oracle.bwd(*args, hi.dy, h0=hi.h0, dhT=hi.dhT, decide=3, on=on)
    for u, v in zip(a, b):
        if u is not None:
            np.testing.assert_array_equal(u, v)
    on0, pre0 = oracle.relu_decisions(2, 7, 4, 16, 32, hi.x, hi.w, h0=hi.h0, decide=0)
    y0, _, _ = oracle.fwd(*args, h0=hi.h0)
    np.testing.assert_array_equal(y0, np.maximum(pre0[1], 0.0))   # top layer output from its pre-activations
    # a decision flipped by hand changes exactly that unit's output at that step
    on2 = on0.copy()
    t, bq, j = np.argwhere(on0[1] == 1)[0]
    on2[1, t, bq, j] = 0
    y2, _, _ = oracle.fwd(*args, h0=hi.h0, decide=3, on=on2)
    assert y2[t, bq, j] == 0.0 and y0[t, bq, j] > 0
    np.testing.assert_array_equal(y2[:t], y0[:t])
