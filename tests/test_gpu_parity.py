"""CUDA path vs the double-precision oracle, element by element, on the same
seeded inputs: tiny shapes of every cell in both storage modes (several
tiles, ragged edges, multi-chunk wavefront), the five benchmark workloads
(in full where the oracle finishes in seconds, otherwise on sampled batch
columns at full size), and the edge cases of the method."""
import numpy as np
import pytest

from recurrent_neural_network_gb300 import rnn, runner, synth

from parity import compare, device_relu_decisions, relu_check, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

TINY = {
    # mode: (L, T, B, I, H)
    synth.MODE_FP32: (2, 5, 3, 40, 64),
    synth.MODE_BF16: (2, 5, 3, 72, 128),
}


def tiny(cell, mode, **kw):
    L, T, B, I, H = TINY[mode]
    base = dict(name="tiny", cell=cell, layers=L, T=T, B=B, input=I, hidden=H, mode=mode,
                forget_bias=1.0, state_std=0.3)
    base.update(kw)
    return synth.Workload(**base)


@pytest.mark.parametrize("mode", [synth.MODE_FP32, synth.MODE_BF16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("cell", [0, 1, 2, 3], ids=["lstm", "gru", "tanh", "relu"])
@pytest.mark.parametrize("chunk", [0, 2], ids=["chunkauto", "chunk2"])
def test_tiny_all_outputs(cell, mode, chunk):
    wl = tiny(cell, mode)
    hi = runner.HostInputs(wl, with_state_grads=True)
    g = run_gpu(wl, hi, chunk=chunk)
    o = run_oracle(hi)
    compare(wl, g, o)


@pytest.mark.parametrize("cell", [0, 1, 2], ids=["lstm", "gru", "tanh"])
def test_layer_by_layer_equals_wavefront(cell):
    wl = tiny(cell, synth.MODE_BF16, layers=3, T=7)
    hi = runner.HostInputs(wl, with_state_grads=True)
    a = run_gpu(wl, hi, chunk=2)
    b = run_gpu(wl, hi, flags=rnn.FLAG_NO_WAVEFRONT)
    for k in a:
        if a[k] is not None:
            np.testing.assert_array_equal(a[k], b[k], err_msg=k)


@pytest.mark.parametrize("cell", [0, 1], ids=["lstm", "gru"])
def test_ragged_batch_and_input(cell):
    """B = 130 spans two 128-row tiles with a ragged tail; I = 72 is not a multiple of 64."""
    wl = synth.Workload("ragged", cell, 2, 3, 130, 72, 128, synth.MODE_BF16, forget_bias=1.0, state_std=0.2)
    hi = runner.HostInputs(wl, with_state_grads=True)
    compare(wl, run_gpu(wl, hi), run_oracle(hi))


@pytest.mark.parametrize("cell,B,H", [(1, 4, 192), (0, 70, 320), (2, 9, 64), (1, 33, 256)],
                         ids=["gru_B4_H192", "lstm_B70_H320", "tanh_B9_H64", "gru_B33_H256"])
def test_backward_split_shapes(cell, B, H):
    """Widths whose gate-gradient K blocks are not a power of two (3*192/64 = 9,
    4*320/64 = 20 ...): the backward step's split-K plan and its cluster reduction."""
    wl = synth.Workload("splits", cell, 2, 4, B, 64, H, synth.MODE_BF16, forget_bias=1.0, state_std=0.2)
    hi = runner.HostInputs(wl, with_state_grads=True)
    compare(wl, run_gpu(wl, hi, flags=rnn.FLAG_FORCE_STREAMING), run_oracle(hi))


def test_single_step_and_single_row():
    wl = synth.Workload("t1b1", 0, 1, 1, 1, 64, 64, synth.MODE_BF16, forget_bias=1.0, state_std=0.5)
    hi = runner.HostInputs(wl, with_state_grads=True)
    compare(wl, run_gpu(wl, hi), run_oracle(hi))


def test_zero_input_zero_state_zero_bias_stays_exactly_zero():
    wl = synth.Workload("zeros", 0, 2, 4, 8, 64, 64, synth.MODE_BF16)
    hi = runner.HostInputs(wl)
    hi.x[:] = 0
    g = run_gpu(wl, hi)
    assert not np.any(g["y"]) and not np.any(g["hT"]) and not np.any(g["cT"])


def test_repeated_calls_are_deterministic():
    wl = tiny(0, synth.MODE_BF16, B=9)
    hi = runner.HostInputs(wl, with_state_grads=True)
    a = run_gpu(wl, hi)
    b = run_gpu(wl, hi, repeat=2)
    for k in a:
        if a[k] is not None:
            np.testing.assert_array_equal(a[k], b[k], err_msg=k)


# ---------------------------------------------------------------- benchmark workloads

def test_workload_lstm_fp32_tiny():
    wl = synth.WORKLOADS[0]
    hi = runner.HostInputs(wl)
    compare(wl, run_gpu(wl, hi), run_oracle(hi))


def test_workload_lstm_h512_training():
    wl = synth.WORKLOADS[1]
    hi = runner.HostInputs(wl)
    compare(wl, run_gpu(wl, hi), run_oracle(hi))


def test_workload_lstm_b4_inference():
    wl = synth.WORKLOADS[2]
    hi = runner.HostInputs(wl)
    compare(wl, run_gpu(wl, hi), run_oracle(hi, train=False))


@pytest.mark.parametrize("flags", [rnn.FLAG_FORCE_STREAMING | rnn.FLAG_FORCE_TRANSPOSED,
                                   rnn.FLAG_FORCE_STREAMING | rnn.FLAG_NO_TRANSPOSED],
                         ids=["transposed", "row_major"])
def test_workload_lstm_b4_inference_streaming(flags):
    """The same 1000-step inference on streaming step launches (graph replay on
    the third call), against the oracle."""
    wl = synth.WORKLOADS[2]
    hi = runner.HostInputs(wl)
    o = run_oracle(hi, train=False)
    for repeat in (1, 3):
        compare(wl, run_gpu(wl, hi, flags=flags, repeat=repeat), o)


def masked_columns_check(wl, cols):
    """Full-size run with dy zero outside `cols`; forward outputs, data
    gradients and weight gradients of those columns against the oracle run on
    them alone (sequences are independent; dW sums over columns)."""
    hi = runner.HostInputs(wl)
    mask = np.zeros(wl.B, bool)
    mask[cols] = True
    hi.dy[:, ~mask] = 0
    g = run_gpu(wl, hi)
    sub = hi.columns(cols)
    o = run_oracle(sub)
    gs = dict(y=g["y"][:, cols], hT=g["hT"][:, cols], cT=None if g["cT"] is None else g["cT"][:, cols],
              dx=g["dx"][:, cols], dh0=g["dh0"][:, cols], dc0=None if g["dc0"] is None else g["dc0"][:, cols],
              dw=g["dw"])
    compare(sub.wl, gs, o)
    # columns without upstream gradient get exactly zero data gradients
    assert not np.any(g["dx"][:, ~mask])


def test_workload_lstm_h4096_sampled_columns():
    masked_columns_check(synth.WORKLOADS[3], [0, 201])


def test_workload_gru_8layer_sampled_columns():
    masked_columns_check(synth.WORKLOADS[4], [5, 31])


def test_workload_relu_4layer_sampled_columns():
    """4-layer ReLU RNN, H=2048, B=256, T=100, ordinary weights.  Over 100 steps
    and 4 layers a few on/off decisions are taken at pre-activations within
    rounding of 0, and each one reroutes gradient paths through time, so the
    gradients are checked with the decisions the device took (every one that
    differs from the oracle's bf16-precision decision must lie within the
    forward bar of 0)."""
    wl = synth.WORKLOADS[5]
    cols = [3, 250]
    hi = runner.HostInputs(wl)
    mask = np.zeros(wl.B, bool)
    mask[cols] = True
    hi.dy[:, ~mask] = 0
    g = run_gpu(wl, hi)
    sub = hi.columns(cols)
    gs = dict(y=g["y"][:, cols], hT=g["hT"][:, cols], cT=None, dx=g["dx"][:, cols], dh0=g["dh0"][:, cols], dc0=None,
              dw=g["dw"])
    on = device_relu_decisions(wl, hi, g, cols=cols)
    relu_check(sub.wl, sub, gs, on)
    assert not np.any(g["dx"][:, ~mask])


def test_workload_bidirectional_lstm_sampled_columns():
    masked_columns_check(synth.WORKLOADS[6], [77])


# ---------------------------------------------------------------- persistent recurrence

PERSIST_CASES = [
    # cell, layers, T, B, I, H
    (0, 1, 7, 1, 64, 128),
    (0, 2, 6, 3, 72, 1024),
    (0, 1, 5, 8, 128, 256),
    (1, 2, 6, 4, 64, 256),
    (1, 1, 5, 8, 64, 128),
    (1, 1, 6, 4, 64, 1024),
    (2, 2, 6, 5, 64, 2048),
    (3, 2, 6, 4, 64, 512),
]


# hand-off variants: tagged words gathered per cluster (default), arrival counters
HANDOFF = [0, rnn.FLAG_PERSIST_CLUSTER_SYNC, rnn.FLAG_NO_PERSIST_CLUSTER]
HANDOFF_IDS = ["cluster_async", "cluster_sync", "counter"]


def persist_cluster_of(r):
    return int(r.r.describe().split("persist_cluster=")[1].split()[0])


@pytest.mark.parametrize("handoff", HANDOFF, ids=HANDOFF_IDS)
@pytest.mark.parametrize("case", PERSIST_CASES, ids=lambda c: "c%d_L%d_T%d_B%d_I%d_H%d" % c)
def test_persistent_recurrence_training(case, handoff):
    cell, L, T, B, I, H = case
    wl = synth.Workload("persist", cell, L, T, B, I, H, synth.MODE_BF16, forget_bias=1.0, state_std=0.3)
    hi = runner.HostInputs(wl, with_state_grads=True)
    fl = rnn.FLAG_FORCE_PERSISTENT | handoff
    r = runner.Runner(wl, flags=fl)
    assert "recurrence=persistent" in r.r.describe()
    # the cluster hand-off is taken where its words fit the pollers (else counters)
    assert (persist_cluster_of(r) == 0) if handoff == rnn.FLAG_NO_PERSIST_CLUSTER else persist_cluster_of(r) in (0, 2, 4, 8)
    compare(wl, run_gpu(wl, hi, flags=fl), run_oracle(hi))


@pytest.mark.parametrize("cell,H,B", [(0, 1024, 4), (1, 512, 8), (2, 2048, 3), (3, 256, 1)])
def test_persistent_handoff_variants_bit_identical(cell, H, B):
    """Every hand-off feeds the same bf16 h_{t-1} to the same arithmetic."""
    wl = synth.Workload("hand", cell, 1, 40, B, 64, H, synth.MODE_BF16, forget_bias=1.0, state_std=0.3)
    hi = runner.HostInputs(wl, with_state_grads=True)
    assert persist_cluster_of(runner.Runner(wl, flags=rnn.FLAG_FORCE_PERSISTENT)) in (2, 4, 8)
    a = run_gpu(wl, hi, flags=rnn.FLAG_FORCE_PERSISTENT)
    for other in (rnn.FLAG_PERSIST_CLUSTER_SYNC, rnn.FLAG_NO_PERSIST_CLUSTER):
        b = run_gpu(wl, hi, flags=rnn.FLAG_FORCE_PERSISTENT | other)
        for k in a:
            if a[k] is not None:
                assert np.array_equal(a[k], b[k]), (other, k)


def test_persistent_equals_streaming_within_tolerance():
    wl = synth.Workload("pvs", 0, 2, 9, 4, 128, 512, synth.MODE_BF16, forget_bias=1.0, state_std=0.3)
    hi = runner.HostInputs(wl, with_state_grads=True)
    p = run_gpu(wl, hi, flags=rnn.FLAG_FORCE_PERSISTENT)
    s = run_gpu(wl, hi, flags=rnn.FLAG_FORCE_STREAMING)
    for k in ("y", "hT", "cT"):
        assert float(np.abs(p[k] - s[k]).max()) <= 3e-2, k


@pytest.mark.parametrize("handoff", HANDOFF, ids=HANDOFF_IDS)
def test_persistent_bounded_wait_reports_timeout(handoff):
    """One CTA never publishes its first step: the others' waits give up after
    the handle's bound and the error word says so; the context stays usable."""
    wl = synth.Workload("skip", 0, 1, 4, 2, 64, 256, synth.MODE_BF16, training=False)
    hi = runner.HostInputs(wl)
    r = runner.Runner(wl, flags=rnn.FLAG_FORCE_PERSISTENT | rnn.FLAG_TEST_SKIP_PUBLISH | handoff,
                      timeout_ns=20_000_000)
    r.upload(hi)
    r.forward(False)
    assert r.status() == -5  # RNN_ERR_TIMEOUT
    assert r.status() == 0   # the word was cleared
    g = run_gpu(wl, hi, flags=rnn.FLAG_FORCE_PERSISTENT)
    compare(wl, g, run_oracle(hi, train=False))


# ---------------------------------------------------------------- graph replay

@pytest.mark.parametrize("flags,kw", [(0, dict(layers=3, T=7, B=9)), (rnn.FLAG_FORCE_PERSISTENT, dict(layers=2, T=6, B=4)),
                                      (0, dict(layers=2, T=5, B=200))], ids=["wavefront", "persistent", "pairs"])
def test_graph_capture_and_replay_match_direct_calls(flags, kw):
    """Call 1 runs directly, call 2 is captured into a CUDA graph and launched,
    call 3 replays it: all three give identical results, equal to a handle that
    never uses graphs."""
    wl = tiny(0, synth.MODE_BF16, **kw)
    hi = runner.HostInputs(wl, with_state_grads=True)
    r = runner.Runner(wl, flags=flags, chunk=2)
    r.upload(hi)
    outs = []
    for _ in range(3):
        r.step()
        assert r.status() == 0
        outs.append(r.outputs())
    ref = run_gpu(wl, hi, flags=flags | rnn.FLAG_NO_GRAPH, chunk=2)
    for o in outs:
        for k in ref:
            if ref[k] is not None:
                np.testing.assert_array_equal(o[k], ref[k], err_msg=k)
    compare(wl, outs[-1], run_oracle(hi))


@pytest.mark.gpu
@pytest.mark.parametrize("cell", [0, 1, 2])
@pytest.mark.parametrize("kw", [dict(layers=3, T=7, B=9, hidden=256), dict(layers=2, T=5, B=200, hidden=256)],
                         ids=["one_cta", "pairs"])
def test_dependent_launch_matches_serialised_launches(cell, kw):
    """Programmatic dependent launch (the default on a single stream of
    launches: here the wavefront is off) lets each tensor-core kernel start
    and load its weights while the previous one drains; the results are
    bit-identical to launches that each wait for their predecessor."""
    wl = tiny(cell, synth.MODE_BF16, **kw)
    hi = runner.HostInputs(wl, with_state_grads=True)
    fl = rnn.FLAG_FORCE_STREAMING | rnn.FLAG_NO_WAVEFRONT
    a = run_gpu(wl, hi, flags=fl)
    b = run_gpu(wl, hi, flags=fl | rnn.FLAG_NO_PDL)
    for k in b:
        if b[k] is not None:
            np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    compare(wl, a, run_oracle(hi))


TRANSPOSED = [
    # (cell, L, T, B, I, H): ragged batch and unit tiles, every batch-tile width, wavefront chunks
    (0, 2, 5, 9, 72, 256),
    (0, 2, 4, 200, 64, 192),
    (0, 1, 3, 64, 128, 128),
    (0, 1, 3, 256, 64, 512),
    (0, 3, 6, 1, 64, 256),
    (0, 2, 4, 129, 72, 320),
    (2, 2, 5, 9, 72, 256),
    (2, 2, 4, 130, 64, 384),
    (3, 2, 5, 9, 72, 256),
    (3, 2, 4, 200, 64, 320),
    (0, 2, 5, 200, 64, 256),   # 256-wide batch tiles, 4 splits: pointwise BPTT fused into the product
    (0, 2, 4, 256, 64, 256),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", TRANSPOSED, ids=[f"c{c}_L{L}_T{T}_B{B}_I{I}_H{H}" for c, L, T, B, I, H in TRANSPOSED])
def test_transposed_steps(case):
    """Recurrent steps taken as W_h h^T (packing unit 1, batch on the tile
    columns) against the oracle, every output and gradient."""
    cell, L, T, B, I, H = case
    wl = synth.Workload(name="transposed", cell=cell, layers=L, T=T, B=B, input=I, hidden=H, mode=synth.MODE_BF16,
                        forget_bias=1.0, state_std=0.3)
    hi = runner.HostInputs(wl, with_state_grads=True)
    g = run_gpu(wl, hi, flags=rnn.FLAG_FORCE_TRANSPOSED | rnn.FLAG_FORCE_STREAMING, chunk=2)
    compare(wl, g, run_oracle(hi))


@pytest.mark.gpu
def test_transposed_equals_row_major_steps_within_tolerance():
    """Both step orientations on the same inputs agree to bf16 rounding; the
    transposed one is deterministic across repeated calls (graph replay)."""
    wl = tiny(0, synth.MODE_BF16, layers=2, T=6, B=33, hidden=256)
    hi = runner.HostInputs(wl, with_state_grads=True)
    a = run_gpu(wl, hi, flags=rnn.FLAG_FORCE_TRANSPOSED | rnn.FLAG_FORCE_STREAMING)
    b = run_gpu(wl, hi, flags=rnn.FLAG_NO_TRANSPOSED | rnn.FLAG_FORCE_STREAMING)
    compare(wl, a, b)
    r = runner.Runner(wl, flags=rnn.FLAG_FORCE_TRANSPOSED | rnn.FLAG_FORCE_STREAMING)
    r.upload(hi)
    outs = []
    for _ in range(3):
        r.step()
        assert r.status() == 0
        outs.append(r.outputs())
    for o in outs[1:]:
        for k in outs[0]:
            if outs[0][k] is not None:
                np.testing.assert_array_equal(o[k], outs[0][k], err_msg=k)


@pytest.mark.gpu
@pytest.mark.parametrize("B", [200, 256])
def test_fused_pointwise_equals_separate_kernel(B):
    """The transposed LSTM BPTT runs its pointwise step inside the product's
    epilogue (inputs staged by bulk loads) or as its own kernel: same
    arithmetic in the same order, bit-identical results."""
    wl = tiny(0, synth.MODE_BF16, layers=2, T=5, B=B, hidden=256)
    hi = runner.HostInputs(wl, with_state_grads=True)
    r = runner.Runner(wl, flags=rnn.FLAG_FORCE_TRANSPOSED | rnn.FLAG_FORCE_STREAMING)
    assert "fused_point=1" in r.r.describe()
    a = run_gpu(wl, hi, flags=rnn.FLAG_FORCE_TRANSPOSED | rnn.FLAG_FORCE_STREAMING)
    b = run_gpu(wl, hi, flags=rnn.FLAG_FORCE_TRANSPOSED | rnn.FLAG_FORCE_STREAMING | rnn.FLAG_NO_FUSED_POINT)
    for k in b:
        if b[k] is not None:
            np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    compare(wl, a, run_oracle(hi))


SLIM = [dict(layers=2, T=5, B=256, hidden=256), dict(layers=2, T=4, B=200, hidden=384),
        dict(layers=1, T=3, B=129, hidden=128), dict(layers=2, T=4, B=256, hidden=256, training=False)]


@pytest.mark.gpu
@pytest.mark.parametrize("kw", SLIM, ids=["B256_H256", "B200_H384", "B129_H128", "B256_H256_infer"])
def test_slim_forward_step_equals_standard(kw):
    """RNN_FLAG_SLIM_STEP: the transposed LSTM forward step on the shared-SM
    kernel (three stages, one TMEM accumulator; P brought in and gates, c and
    h sent out by 16-row bulk copies through a ring of slots) does the same
    arithmetic in the same order as the standard step: bit-identical outputs
    and gradients (ragged last slices included), and the oracle's."""
    wl = tiny(0, synth.MODE_BF16, **kw)
    train = kw.get("training", True)
    hi = runner.HostInputs(wl, with_state_grads=train)
    fl = rnn.FLAG_FORCE_TRANSPOSED | rnn.FLAG_FORCE_STREAMING
    assert "slim_step=1" in runner.Runner(wl, flags=fl | rnn.FLAG_SLIM_STEP).r.describe()
    a = run_gpu(wl, hi, flags=fl | rnn.FLAG_SLIM_STEP)
    b = run_gpu(wl, hi, flags=fl)
    for k in b:
        if b[k] is not None:
            np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    compare(wl, a, run_oracle(hi, train=train))


CHUNKS = [(dict(layers=2, T=9, B=256, hidden=256), 4), (dict(layers=3, T=8, B=96, hidden=384), 8),
          (dict(layers=1, T=6, B=64, hidden=128), 0), (dict(layers=2, T=7, B=160, hidden=1024), 4)]


@pytest.mark.gpu
@pytest.mark.parametrize("kw,chunk", CHUNKS, ids=["B256_H256_c4", "B96_H384_c8", "B64_H128_L1", "B160_H1024_c4"])
def test_step_chunks_equal_step_launches(kw, chunk):
    """RNN_FLAG_STEP_CHUNKS: the transposed LSTM training steps of a chunk
    after t = 0 in one cooperative launch (each CTA pair loads h_{t-1} once
    every pair has stored it, and c_{t-1} comes from its own stores) do the
    same arithmetic in the same order as one launch per step: bit-identical
    outputs, final states and gradients (single-step chunks, the last step
    inside a multi-step launch, tiles wider than the batch), and the
    oracle's."""
    wl = tiny(0, synth.MODE_BF16, **kw)
    hi = runner.HostInputs(wl, with_state_grads=True)
    fl = rnn.FLAG_FORCE_TRANSPOSED | rnn.FLAG_FORCE_STREAMING
    assert "step_chunks=1" in runner.Runner(wl, flags=fl | rnn.FLAG_STEP_CHUNKS, chunk=chunk).r.describe()

    def fwd_launches(flags):
        r = runner.Runner(wl, flags=flags | rnn.FLAG_NO_GRAPH, chunk=chunk)
        r.upload(hi)
        n0 = rnn.launch_count()
        r.forward(True)
        assert r.status() == 0
        return rnn.launch_count() - n0

    # the steps of a chunk after t = 0 really run as one launch
    assert fwd_launches(fl | rnn.FLAG_STEP_CHUNKS) < fwd_launches(fl)
    a = run_gpu(wl, hi, flags=fl | rnn.FLAG_STEP_CHUNKS, chunk=chunk, repeat=2)
    b = run_gpu(wl, hi, flags=fl, chunk=chunk)
    for k in b:
        if b[k] is not None:
            np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    compare(wl, a, run_oracle(hi))


@pytest.mark.gpu
@pytest.mark.parametrize("flags,B", [(rnn.FLAG_FORCE_STREAMING | rnn.FLAG_NO_TRANSPOSED, 33),
                                     (rnn.FLAG_FORCE_TRANSPOSED | rnn.FLAG_FORCE_STREAMING, 33),
                                     (rnn.FLAG_FORCE_PERSISTENT, 4),
                                     (rnn.FLAG_FORCE_PERSISTENT | rnn.FLAG_NO_PERSIST_CLUSTER, 4)],
                         ids=["row_major", "transposed", "persistent", "persistent_counter"])
def test_relu_training_with_ordinary_weights(flags, B):
    """ReLU RNN with the ordinary weight distribution (pre-activations cross 0
    everywhere): every output and gradient against the oracle, which takes each
    unit's on/off decision as a device storing h in bf16 does (the values stay
    double), and against the oracle run with the decisions the device took."""
    wl = synth.Workload(name="relu", cell=3, layers=2, T=6, B=B, input=72, hidden=256, mode=synth.MODE_BF16,
                        state_std=0.3)
    hi = runner.HostInputs(wl, with_state_grads=True)
    g = run_gpu(wl, hi, flags=flags)
    # with the oracle deciding in bf16 precision the gradients agree as they are
    compare(wl, g, run_oracle(hi))
    # and exactly so with the device's own decisions, which differ from the
    # oracle's only at pre-activations within the forward bar of 0
    relu_check(wl, hi, g, device_relu_decisions(wl, hi, g, flags=flags))


# ---------------------------------------------------------------- variable lengths

VARLEN = [
    # cell, mode, flags, (L, T, B, I, H)
    (0, synth.MODE_BF16, 0, (2, 7, 9, 72, 128)),
    (0, synth.MODE_BF16, rnn.FLAG_FORCE_TRANSPOSED | rnn.FLAG_FORCE_STREAMING, (2, 7, 9, 72, 256)),
    (0, synth.MODE_BF16, rnn.FLAG_FORCE_TRANSPOSED | rnn.FLAG_FORCE_STREAMING, (2, 6, 200, 64, 256)),
    (1, synth.MODE_BF16, 0, (2, 7, 9, 72, 128)),
    (2, synth.MODE_BF16, 0, (2, 7, 9, 72, 128)),
    (3, synth.MODE_BF16, rnn.FLAG_FORCE_TRANSPOSED | rnn.FLAG_FORCE_STREAMING, (2, 7, 9, 72, 256)),
    (0, synth.MODE_FP32, 0, (2, 7, 5, 40, 64)),
    (1, synth.MODE_FP32, 0, (2, 7, 5, 40, 64)),
    (0, synth.MODE_BF16, 0, (1, 9, 4, 64, 256)),   # planned persistent: switches to step launches
]


def _lengths(T, B, seed):
    rng = np.random.default_rng(seed)
    lens = np.sort(rng.integers(1, T + 1, size=B))[::-1].copy()
    lens[0] = T
    return [int(v) for v in lens]


@pytest.mark.gpu
@pytest.mark.parametrize("case", VARLEN, ids=lambda c: "c%d_m%d_f%x_L%d_T%d_B%d_I%d_H%d" % (c[0], c[1], c[2], *c[3]))
def test_variable_lengths(case):
    """Sequences of different lengths (sorted longest first) against the
    oracle with the same lengths: outputs zero past each end, final states
    after each sequence's own last step, every gradient; twice through the
    same handle (direct call, then the captured graph)."""
    cell, mode, flags, (L, T, B, I, H) = case
    wl = synth.Workload(name="varlen", cell=cell, layers=L, T=T, B=B, input=I, hidden=H, mode=mode,
                        forget_bias=1.0, state_std=0.3)
    hi = runner.HostInputs(wl, with_state_grads=True)
    lens = _lengths(T, B, seed=B + T + cell)
    g = run_gpu(wl, hi, flags=flags, chunk=2, lens=lens, repeat=2)
    o = run_oracle(hi, lens=lens)
    compare(wl, g, o)
    for b, n in enumerate(lens):
        assert not np.any(g["y"][n:, b]), b
        assert not np.any(g["dx"][n:, b]), b


# ---------------------------------------------------------------- bidirectional layers

BIDIR = [
    # cell, mode, flags, (L, T, B, I, H)
    (0, synth.MODE_BF16, 0, (2, 7, 9, 72, 128)),                              # row-major steps
    (0, synth.MODE_BF16, rnn.FLAG_FORCE_TRANSPOSED, (2, 6, 9, 72, 256)),      # transposed, separate pointwise
    (0, synth.MODE_BF16, rnn.FLAG_FORCE_TRANSPOSED, (2, 5, 200, 64, 256)),    # transposed, fused pointwise
    (1, synth.MODE_BF16, 0, (2, 6, 9, 72, 128)),
    (2, synth.MODE_BF16, 0, (3, 5, 9, 72, 128)),
    (3, synth.MODE_BF16, rnn.FLAG_FORCE_TRANSPOSED, (2, 6, 9, 72, 256)),
    (0, synth.MODE_FP32, 0, (2, 5, 5, 40, 64)),
    (1, synth.MODE_FP32, 0, (2, 5, 5, 40, 64)),
    (2, synth.MODE_FP32, 0, (1, 4, 3, 36, 32)),
    (0, synth.MODE_BF16, rnn.FLAG_NO_WAVEFRONT, (2, 6, 9, 72, 128)),        # directions one after the other
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", BIDIR, ids=lambda c: "c%d_m%d_f%x_L%d_T%d_B%d_I%d_H%d" % (c[0], c[1], c[2], *c[3]))
def test_bidirectional(case):
    """Bidirectional stacks against the oracle: y = [forward, reverse] per
    timestep, final states and their gradients per (layer, direction), dx and
    every weight block; twice through the same handle (direct call, then the
    captured graph)."""
    cell, mode, flags, (L, T, B, I, H) = case
    wl = synth.Workload(name="bidir", cell=cell, layers=L, T=T, B=B, input=I, hidden=H, mode=mode,
                        forget_bias=1.0, state_std=0.3, directions=2)
    hi = runner.HostInputs(wl, with_state_grads=True)
    g = run_gpu(wl, hi, flags=flags, repeat=2)
    compare(wl, g, run_oracle(hi))


@pytest.mark.gpu
def test_bidirectional_inference_matches_training_forward():
    wl = synth.Workload(name="bidir", cell=0, layers=2, T=6, B=9, input=72, hidden=128, mode=synth.MODE_BF16,
                        forget_bias=1.0, state_std=0.3, directions=2)
    hi = runner.HostInputs(wl)
    a = run_gpu(wl.replace(training=False), hi)
    b = run_gpu(wl, hi, train=True)
    for k in ("y", "hT", "cT"):
        assert np.array_equal(a[k], b[k]), k


BIDIR_VARLEN = [
    # cell, mode, flags, (L, T, B, I, H)
    (0, synth.MODE_BF16, 0, (2, 7, 9, 72, 128)),
    (0, synth.MODE_BF16, rnn.FLAG_FORCE_TRANSPOSED, (2, 7, 9, 72, 256)),
    (0, synth.MODE_BF16, rnn.FLAG_FORCE_TRANSPOSED, (2, 6, 200, 64, 256)),
    (1, synth.MODE_BF16, 0, (2, 7, 9, 72, 128)),
    (2, synth.MODE_BF16, 0, (2, 7, 9, 72, 128)),
    (3, synth.MODE_BF16, rnn.FLAG_FORCE_TRANSPOSED, (2, 7, 9, 72, 256)),
    (0, synth.MODE_FP32, 0, (2, 7, 5, 40, 64)),
    (1, synth.MODE_FP32, 0, (2, 7, 5, 40, 64)),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", BIDIR_VARLEN, ids=lambda c: "c%d_m%d_f%x_L%d_T%d_B%d_I%d_H%d" % (c[0], c[1], c[2], *c[3]))
def test_bidirectional_variable_lengths(case):
    """Bidirectional stacks with sequences of different lengths: the reverse
    sweep of each sequence starts at its own last step from its h0; y is zero
    past each end in both halves; every gradient against the oracle; twice
    through the same handle."""
    cell, mode, flags, (L, T, B, I, H) = case
    wl = synth.Workload(name="bivar", cell=cell, layers=L, T=T, B=B, input=I, hidden=H, mode=mode,
                        forget_bias=1.0, state_std=0.3, directions=2)
    hi = runner.HostInputs(wl, with_state_grads=True)
    lens = _lengths(T, B, seed=3 * B + T + cell)
    g = run_gpu(wl, hi, flags=flags, lens=lens, repeat=2)
    compare(wl, g, run_oracle(hi, lens=lens))
    for b, n in enumerate(lens):
        assert not np.any(g["y"][n:, b]), b
        assert not np.any(g["dx"][n:, b]), b


PERSIST_BIDIR = [
    # cell, layers, T, B, I, H
    (0, 2, 6, 4, 64, 256),
    (0, 1, 40, 4, 64, 1024),
    (1, 2, 5, 8, 64, 128),
    (2, 1, 7, 3, 64, 512),
    (3, 2, 6, 4, 64, 256),
]


@pytest.mark.gpu
@pytest.mark.parametrize("handoff", HANDOFF, ids=HANDOFF_IDS)
@pytest.mark.parametrize("case", PERSIST_BIDIR, ids=lambda c: "c%d_L%d_T%d_B%d_I%d_H%d" % c)
def test_bidirectional_persistent_recurrence(case, handoff):
    """Small-batch bidirectional stacks on the persistent recurrence (one launch
    per direction, the reverse one walking time backwards), training against
    the oracle with both hand-offs."""
    cell, L, T, B, I, H = case
    wl = synth.Workload("pbidir", cell, L, T, B, I, H, synth.MODE_BF16, forget_bias=1.0, state_std=0.3,
                        directions=2)
    hi = runner.HostInputs(wl, with_state_grads=True)
    fl = rnn.FLAG_FORCE_PERSISTENT | handoff
    assert "recurrence=persistent" in runner.Runner(wl, flags=fl).r.describe()
    compare(wl, run_gpu(wl, hi, flags=fl, repeat=2), run_oracle(hi))
