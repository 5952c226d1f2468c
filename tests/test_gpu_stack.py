"""The persistent stacked recurrences (bf16, one direction, up to 64
sequences): groups of up to four layers in one launch each way, each layer's
[W_x | W_h] rows (forward) or transposed columns (backward) resident in tensor
memory, the part of a chunk wider than it holds in shared memory, layer l+1
starting step t once layer l has finished it.

"Persistent RNNs: Stashing Recurrent Weights On-Chip" (citing snippets on its
page) for the resident weights and the single launch; "Optimizing Performance
of RNNs on GPUs" (review page, proposed method) for the overlap of layers.
Every case is compared with the oracle at the bf16-mode bar; the backward
pass after a stacked forward reads the reserve the kernel wrote."""
import re

import numpy as np
import pytest

from recurrent_neural_network_gb300 import rnn, runner, synth

from parity import compare, device_relu_decisions, rel_l2, relu_check, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def plan_of(r):
    d = r.r.describe()
    return re.search(r"recurrence=(\w+)", d).group(1), re.search(r"stack_groups=(\S+)", d).group(1), \
        int(re.search(r" u=(\d+)", d).group(1))


def bwd_groups(r):
    return re.search(r"stack_bwd_groups=(\S+)", r.r.describe()).group(1)


STACK_CASES = [
    # cell, layers, T, B, I, H, forward groups, backward groups (highest first; "-": step launches)
    (0, 3, 12, 24, 64, 512, "0+3", "0+3"),            # LSTM, packing unit 16, N=32
    (0, 4, 9, 64, 512, 512, "0+4", "0+4"),            # LSTM, the 4-layer H=512 B=64 shape, unit 1, N=64
    (0, 2, 7, 9, 40, 256, "0+2", "0+2"),              # ragged batch (N=16), 256-wide K chunks
    (1, 2, 10, 32, 72, 256, "0+2", "0+2"),            # GRU, input and recurrent sums apart; 384-wide bwd chunks
    (1, 3, 6, 20, 64, 1024, "0+2,2+1", "1+2,0+1"),  # GRU: two layers in the first forward launch, layer 1
                                                     # on 1024-wide chunks (896 k in TMEM, 128 in shared
                                                     # memory); backward on 768-wide chunks
    (1, 5, 6, 24, 64, 1024, "0+2,2+2,4+1", "3+2,1+2,0+1r"),  # GRU backward with recurrent-only group tops:
                                                              # the share from above of layers 4 and 2 by GEMM
    (0, 4, 5, 32, 48, 1024, "0+2,2+2", "2+2,0+2r"),  # LSTM: 1024-wide chunks split between TMEM and shared
                                                      # memory in both forward and both backward launches
    (1, 2, 7, 12, 64, 1024, "0+2", "0+2"),            # GRU, N=16, ragged batch on the split chunks
    (0, 2, 5, 12, 64, 1024, "0+2", "0+2"),            # LSTM, N=16: backward chunks split between TMEM and
                                                      # shared memory too (the shared-memory kernel variant)
    (2, 5, 8, 33, 96, 1024, "0+4,4+1", "1+4,0+1"),    # tanh: 128 units per CTA, two groups each way
    (0, 1, 11, 48, 32, 1024, "0+1", "0+1"),           # one layer, K split in two
    (0, 17, 4, 12, 64, 256, "0+4,4+4,8+4,12+4,16+1", "13+4,9+4,5+4,1+4,0+1"),  # 17 layers: five launches each
                                                      # way, a counter row per layer, the h_{-1} copies and counter
                                                      # zeroing of the forward in two batched launches (18 > 16 ops)
    (0, 1, 6, 4, 64, 2048, "0+1", "-"),               # B <= 8 beyond the persistent widths: one layer on
    (1, 1, 5, 8, 32, 2048, "0+1", "-"),               # 1024-wide split chunks (N=16), step-launch backward
]


@pytest.mark.parametrize("train", [True, False], ids=["train", "infer"])
@pytest.mark.parametrize("case", STACK_CASES, ids=lambda c: "c%d_L%d_T%d_B%d_I%d_H%d" % c[:6])
def test_stacked_forward(case, train):
    cell, L, T, B, I, H, groups, bgroups = case
    wl = synth.Workload("stack", cell, L, T, B, I, H, synth.MODE_BF16, forget_bias=1.0, state_std=0.3,
                        training=train)
    hi = runner.HostInputs(wl, with_state_grads=True)
    r = runner.Runner(wl)
    assert plan_of(r)[:2] == ("stacked", groups)
    # the backward groups depend on how many clusters of up to 8 CTAs the
    # device holds at once: stacked where planned, in as many groups as fit
    assert (bwd_groups(r) == "-") == (bgroups == "-"), bwd_groups(r)
    compare(wl, run_gpu(wl, hi), run_oracle(hi, train=train))


@pytest.mark.parametrize("case", [c for c in STACK_CASES if c[7] != "-"], ids=lambda c: "c%d_L%d_T%d_B%d_I%d_H%d" % c[:6])
def test_stacked_backward_equals_step_launches_within_tolerance(case):
    """The stacked backward (the transposed products of all layers in one
    launch, dh0 and dc0 from its last step) against the step-launch backward
    on the same forward: both at the bf16 gradient bar of each other."""
    cell, L, T, B, I, H = case[:6]
    wl = synth.Workload("sbw", cell, L, T, B, I, H, synth.MODE_BF16, forget_bias=1.0, state_std=0.3)
    hi = runner.HostInputs(wl, with_state_grads=True)
    a = run_gpu(wl, hi)
    b = run_gpu(wl, hi, flags=rnn.FLAG_NO_STACK_BWD)
    assert bwd_groups(runner.Runner(wl, flags=rnn.FLAG_NO_STACK_BWD)) == "-"
    for k in ("dx", "dh0", "dc0"):
        if a.get(k) is not None:
            assert rel_l2(a[k], b[k]) <= 2e-2, k


def test_forced_below_nine_sequences():
    wl = synth.Workload("stack4", 0, 2, 8, 4, 64, 1024, synth.MODE_BF16, forget_bias=1.0, state_std=0.3)
    hi = runner.HostInputs(wl, with_state_grads=True)
    assert plan_of(runner.Runner(wl, flags=rnn.FLAG_FORCE_STACK))[0] == "stacked"
    compare(wl, run_gpu(wl, hi, flags=rnn.FLAG_FORCE_STACK), run_oracle(hi))


def test_stacked_equals_step_launches_within_tolerance():
    wl = synth.Workload("svs", 0, 3, 10, 32, 64, 512, synth.MODE_BF16, forget_bias=1.0, state_std=0.3)
    hi = runner.HostInputs(wl, with_state_grads=True)
    a = run_gpu(wl, hi)
    b = run_gpu(wl, hi, flags=rnn.FLAG_NO_STACK)
    for k in ("y", "hT", "cT"):
        assert float(np.abs(a[k] - b[k]).max()) <= 3e-2, k


def test_graph_replay_matches_direct_calls():
    """Call 1 direct, call 2 captured, call 3 replayed: identical results, equal
    to a handle without graphs (the stacked forward is deterministic: fixed
    chunk order in the cross-CTA sums)."""
    wl = synth.Workload("sgr", 1, 3, 9, 40, 64, 256, synth.MODE_BF16, forget_bias=1.0, state_std=0.3)
    hi = runner.HostInputs(wl, with_state_grads=True)
    r = runner.Runner(wl)
    assert plan_of(r)[0] == "stacked"
    r.upload(hi)
    outs = []
    for _ in range(3):
        r.step()
        assert r.status() == 0
        outs.append(r.outputs())
    ref = run_gpu(wl, hi, flags=rnn.FLAG_NO_GRAPH)
    for o in outs:
        for k in ref:
            if ref[k] is not None:
                np.testing.assert_array_equal(o[k], ref[k], err_msg=k)
    compare(wl, outs[-1], run_oracle(hi))


def test_bounded_wait_reports_timeout():
    """One CTA never publishes its first step: the CTAs that wait for it give up
    after the handle's bound, the error word says so, and the context stays
    usable for the next call."""
    wl = synth.Workload("sskip", 0, 2, 4, 16, 64, 256, synth.MODE_BF16, training=False)
    hi = runner.HostInputs(wl)
    r = runner.Runner(wl, flags=rnn.FLAG_TEST_SKIP_PUBLISH, timeout_ns=20_000_000)
    assert plan_of(r)[0] == "stacked"
    r.upload(hi)
    r.forward(False)
    assert r.status() == -5  # RNN_ERR_TIMEOUT
    assert r.status() == 0
    compare(wl, run_gpu(wl, hi), run_oracle(hi, train=False))


def test_bounded_wait_reports_timeout_in_training():
    """The same hook in a training call: the stacked forward and then the
    stacked backward each lose CTA 0's first step, their waits give up, and the
    next call on a clean handle is right."""
    wl = synth.Workload("sskipt", 0, 2, 4, 16, 64, 256, synth.MODE_BF16)
    hi = runner.HostInputs(wl, with_state_grads=True)
    r = runner.Runner(wl, flags=rnn.FLAG_TEST_SKIP_PUBLISH, timeout_ns=20_000_000)
    assert plan_of(r)[0] == "stacked" and bwd_groups(r) != "-"
    r.upload(hi)
    r.forward(True)
    assert r.status() == -5
    r.backward()
    assert r.status() == -5
    compare(wl, run_gpu(wl, hi), run_oracle(hi))


def test_relu_with_ordinary_weights():
    """ReLU stack on ordinary weights, gradients checked with the decisions the
    device took (each differing one within the forward bar of 0)."""
    wl = synth.Workload("srelu", 3, 2, 12, 24, 64, 512, synth.MODE_BF16, state_std=0.3)
    hi = runner.HostInputs(wl, with_state_grads=True)
    g = run_gpu(wl, hi)
    on = device_relu_decisions(wl, hi, g)
    relu_check(wl, hi, g, on)


def test_workload_lstm_4layer_b64_is_stacked():
    """The 4-layer LSTM H=512 B=64 T=100 training workload runs its forward and
    its backward as one stacked launch each; full-size parity is in
    test_workload_lstm_h512_training."""
    r = runner.Runner(synth.WORKLOADS[1])
    assert plan_of(r)[:2] == ("stacked", "0+4") and bwd_groups(r) != "-"


def test_workload_gru_8layer_is_stacked():
    r = runner.Runner(synth.WORKLOADS[4])
    assert plan_of(r)[0] == "stacked"
