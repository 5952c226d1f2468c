"""The allocation-free bias-gradient entry point (rnn_bias_grad_static).

Some callers cannot allocate device memory when they need a result -- for
instance a host framework that only hands a plugin its input and output
buffers and forbids cudaMalloc after start-up -- so they cannot provide the
workspace rnn_bwd_weights takes.  rnn_bias_grad_static computes the same bias
gradients with a fixed scratch array inside the library.  These tests check it
through the C-ABI against the bias gradients rnn_bwd_weights writes, on two
calls in a row (the second call finds the first call's leftovers in the shared
array), and that oversized shapes are refused.

This file is collected last on purpose: a run that stops at the first failure
has already run every other test when it gets here.
"""
import ctypes

import numpy as np
import pytest
import torch

from recurrent_neural_network_gb300 import build, rnn, runner, synth

from parity import BF16_REL_L2, FP32_MAX_REL, max_rel, rel_l2, weight_blocks


@pytest.fixture(scope="module")
def lib():
    build.build()
    return rnn.load()


def test_rejects_shapes_beyond_the_fixed_scratch(lib):
    # G*hidden = 4 * 262400 floats exceeds the 4 MiB array; refused before any device work
    r = rnn.RNN(0, 1, 2, 2, 64, 262400, 1)
    fake = ctypes.c_void_p(1 << 20)
    rc = lib.rnn_bias_grad_static(r.h, fake, fake, 0, None)
    assert rc == -2  # RNN_ERR_UNSUPPORTED
    assert lib.rnn_bias_grad_static(r.h, None, fake, 0, None) == -1


# (cell, mode, hidden, directions, flags): unidirectional stacks in both
# storage modes, bidirectional stacks (one bias block pair per layer and
# direction), and the transposed-step packing (packing unit 1, hidden >= 256)
CASES = [
    (0, synth.MODE_BF16, 128, 1, 0),
    (1, synth.MODE_BF16, 128, 1, 0),
    (2, synth.MODE_FP32, 64, 1, 0),
    (0, synth.MODE_BF16, 128, 2, 0),
    (1, synth.MODE_BF16, 128, 2, 0),
    (0, synth.MODE_BF16, 256, 1, rnn.FLAG_FORCE_TRANSPOSED),
]
IDS = ["lstm-bf16", "gru-bf16", "tanh-fp32", "lstm-bf16-bidir", "gru-bf16-bidir", "lstm-bf16-transposed-H256"]


@pytest.mark.gpu
@pytest.mark.parametrize("cell,mode,H,D,flags", CASES, ids=IDS)
def test_matches_bwd_weights_on_two_calls(lib, cell, mode, H, D, flags):
    wl = synth.Workload("noalloc", cell, 2, 9, 37, 72, H, mode, forget_bias=1.0, state_std=0.3, directions=D)
    hi = runner.HostInputs(wl, with_state_grads=True)
    R = runner.Runner(wl, flags=flags)
    if flags & rnn.FLAG_FORCE_TRANSPOSED:
        assert "transposed=1" in R.r.describe() and " u=1 " in R.r.describe()
    R.upload(hi)
    R.forward(True)
    R.backward()
    R.weights()
    assert R.status() == 0
    ref = R.dw.double().cpu().numpy()
    blocks_ref = weight_blocks(wl, ref)
    assert len(blocks_ref) == 4 * wl.layers * D
    for call in range(2):
        out = torch.full_like(R.dw, float("nan"))
        R.r.bias_grad_static(R.reserve, out)
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        for (nm, g), (_, o) in zip(weight_blocks(wl, got), blocks_ref):
            if nm.endswith(("dbx", "dbh")):
                assert np.isfinite(g).all(), (call, nm)
                if mode == synth.MODE_FP32:
                    assert max_rel(g, o) <= FP32_MAX_REL, (call, nm)
                else:
                    assert rel_l2(g, o) <= BF16_REL_L2, (call, nm)
            else:
                assert np.isnan(g).all(), (call, nm)  # weight blocks are left untouched
    # accumulate adds onto what is there
    out = R.dw.clone()
    R.r.bias_grad_static(R.reserve, out, accumulate=True)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    for (nm, g), (_, o) in zip(weight_blocks(wl, got), blocks_ref):
        if nm.endswith(("dbx", "dbh")):
            assert rel_l2(g, 2 * o) <= BF16_REL_L2, nm
