"""The fp8 stash of the persistent recurrence (RNN_FLAG_FP8_STASH): W_h kept on
chip as e4m3 bytes with one float scale per gate row.

"Persistent RNNs: Stashing Recurrent Weights On-Chip" (citing snippets on its
page): on-chip storage is limited in size and precision, so a lower-precision
copy of the recurrent weights lets wider layers stay resident.  The stash is a
deliberate approximation: the forward pass computes with
W_h' = e4m3(W_h / s) * s, s = max|row| / 448.  Parity is therefore checked in
two parts:

* the quantiser itself, byte for byte, against torch's float8_e4m3fn
  conversion of the same fp32 quotients (integer work: bit-exact);
* the recurrence against the oracle run on the dequantised weights W_h'
  (computed here, independently of the CUDA path), at the bf16-mode bar
  (max abs error 3e-2 on y, hT, cT);
* and, as a stated tolerance of the approximation, the same outputs against
  the oracle on the original weights: max abs error <= 0.1 (e4m3 keeps 3
  mantissa bits, a relative rounding error of at most 2^-4 per weight; for
  W ~ U(+-1/sqrt(H)) that moves a pre-activation by about 0.6% of its spread).
"""
import numpy as np
import pytest
import torch

import oracle
from recurrent_neural_network_gb300 import rnn, runner, synth

from parity import BF16_MAX_ABS, run_gpu

pytestmark = pytest.mark.gpu

FP8_WEIGHT_TOL = 0.1


def quantise_rows(w):
    """(dequantised rows, codes, scales) of a float64 [rows][cols] array of bf16
    values: the scale and the quotients in float32, rounded to e4m3 by torch."""
    w32 = np.asarray(w, np.float32)
    amax = np.abs(w32).max(axis=1)
    s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    v = (w32 / s[:, None]).astype(np.float32)
    q = torch.from_numpy(v).to(torch.float8_e4m3fn)
    deq = q.to(torch.float64).numpy() * s.astype(np.float64)[:, None]
    return deq, q.view(torch.uint8).numpy(), s


def dequantised_inputs(hi):
    """A copy of the host inputs with every W_h replaced by its fp8-stash value."""
    wl = hi.wl
    out = object.__new__(type(hi))
    out.__dict__.update(hi.__dict__)
    out.w = hi.w.copy()
    for (wx, wh, bx, bh) in oracle.split_weights(wl.cell, wl.layers, wl.input, wl.hidden, out.w, D=wl.directions):
        wh[...] = quantise_rows(wh)[0]
    return out


def test_quantiser_is_bit_exact():
    rng = np.random.default_rng(7)
    rows, cols = 300, 512
    w = rng.normal(0, 0.05, (rows, cols))
    w[3] = 0.0                                  # all-zero row: scale 1, codes 0
    w[4] *= 1e-4                                # small values: subnormal codes after scaling
    w[5, 17] = 40.0                             # one large value dominating its row
    w[6] = rng.uniform(-1, 1, cols) * 2.0 ** -130  # below the bf16 normal range
    wb = torch.from_numpy(w).to(torch.bfloat16)
    ref_deq, ref_q, ref_s = quantise_rows(wb.to(torch.float64).numpy())
    dev = torch.device("cuda")
    q = torch.empty(rows, cols, dtype=torch.uint8, device=dev)
    s = torch.empty(rows, dtype=torch.float32, device=dev)
    rnn.quantize_e4m3_rows(wb.to(dev), q, s)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(s.cpu().numpy(), ref_s)
    np.testing.assert_array_equal(q.cpu().numpy(), ref_q)
    assert not q[3].any() and s[3].item() == 1.0


CASES = [
    # cell, layers, T, B, I, H, flags
    (0, 1, 16, 4, 64, 2048, 0),                          # beyond the bf16 register stash (16 units per CTA)
    (1, 2, 8, 8, 64, 2048, 0),                           # GRU at twice the bf16 width
    (0, 2, 10, 3, 72, 256, 0),
    (0, 2, 10, 3, 72, 256, rnn.FLAG_NO_PERSIST_CLUSTER),  # counter hand-off
    (2, 1, 12, 5, 64, 1024, 0),
    (3, 1, 12, 2, 64, 512, 0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "c%d_L%d_T%d_B%d_I%d_H%d_f%x" % c)
def test_fp8_stash_inference(case):
    cell, L, T, B, I, H, flags = case
    wl = synth.Workload(name="fp8", cell=cell, layers=L, T=T, B=B, input=I, hidden=H, mode=synth.MODE_BF16,
                        forget_bias=1.0, state_std=0.3, training=False)
    hi = runner.HostInputs(wl)
    r = runner.Runner(wl, flags=flags | rnn.FLAG_FP8_STASH)
    assert "fp8_stash=1" in r.r.describe()
    r.upload(hi)
    r.forward(False)
    assert r.status() == 0
    g = r.outputs()
    hq = dequantised_inputs(hi)
    y, hT, cT = oracle.fwd(cell, L, T, B, I, H, hq.x, hq.w, h0=hq.h0, c0=hq.c0)
    y0, hT0, cT0 = oracle.fwd(cell, L, T, B, I, H, hi.x, hi.w, h0=hi.h0, c0=hi.c0)
    for name, a, o, o0 in (("y", g["y"], y, y0), ("hT", g["hT"], hT, hT0), ("cT", g["cT"], cT, cT0)):
        if o is None:
            continue
        err = float(np.abs(a - o).max())
        assert err <= BF16_MAX_ABS, (name, err)
        dev = float(np.abs(a - o0).max())
        assert dev <= FP8_WEIGHT_TOL, (name, dev)


def test_fp8_stash_training_calls_keep_the_bf16_weights():
    """With the flag, a training forward runs on the bf16 W_h exactly as without it."""
    wl = synth.Workload(name="fp8t", cell=0, layers=2, T=6, B=4, input=64, hidden=256, mode=synth.MODE_BF16,
                        forget_bias=1.0, state_std=0.3)
    hi = runner.HostInputs(wl)
    a = run_gpu(wl, hi, flags=rnn.FLAG_FP8_STASH)
    b = run_gpu(wl, hi)
    for k in a:
        if a[k] is not None:
            np.testing.assert_array_equal(a[k], b[k], err_msg=k)
