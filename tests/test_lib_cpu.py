"""Host-side checks of librnn that need no GPU: it builds, loads, exports every
symbol include/rnn.h declares, plans buffer sizes, and rejects bad arguments
before touching a device."""
import ctypes
import os
import re

import pytest

from recurrent_neural_network_gb300 import build, rnn, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return rnn.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "rnn.h")).read()
    return sorted(set(re.findall(r"RNN_API\s+[\w\s\*]+?\b(rnn_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) >= 13
    assert set(names) == set(rnn.SYMBOLS)
    for n in names:
        assert hasattr(lib, n), n


def test_strerror(lib):
    assert lib.rnn_strerror(0) == b"ok"
    assert lib.rnn_strerror(-5).startswith(b"a bounded")


def test_rejects_bad_descriptors(lib):
    ok = dict(cell=0, layers=1, T=4, B=2, input=64, hidden=64, mode=1)
    for bad in [dict(cell=4), dict(cell=-1), dict(layers=0), dict(T=0), dict(B=0), dict(hidden=0), dict(mode=2)]:
        d = dict(ok, **bad)
        with pytest.raises(rnn.RnnError) as e:
            rnn.RNN(**d)
        assert e.value.code == -1
    for unsup in [dict(hidden=96), dict(input=12), dict(mode=0, hidden=48)]:
        with pytest.raises(rnn.RnnError) as e:
            rnn.RNN(**dict(ok, **unsup))
        assert e.value.code == -2
    with pytest.raises(rnn.RnnError):
        rnn.RNN(**ok, flags=rnn.FLAG_FORCE_PERSISTENT | rnn.FLAG_FORCE_STREAMING)


@pytest.mark.parametrize("wl", synth.WORKLOADS, ids=lambda w: w.name)
def test_buffer_sizes_cover_the_layouts(lib, wl):
    r = rnn.RNN.for_workload(wl)
    s = r.sizes()
    e = 2 if wl.mode == 1 else 4
    assert s["user_weights"] == wl.weight_count() * e
    G, L, T, B, H, D = wl.G, wl.layers, wl.T, wl.B, wl.hidden, wl.directions
    # reserve holds at least: gates (f32) + h sequence (T+1 slots) + gate gradients, per (layer, direction)
    floor = L * D * (T * B * G * H * 4 + (T + 1) * B * H * e + T * B * G * H * e)
    assert s["reserve"] >= floor
    mats = D * sum(G * H * (wl.in_size(l) + H) for l in range(L))
    assert s["packed_weights"] >= mats * e + L * D * G * H * 4   # matrices in storage type + float biases
    # the wavefront overlaps unidirectional layers; bidirectional ones overlap their directions instead
    assert "wavefront=%d" % (1 if L > 1 and D == 1 else 0) in r.describe()
    assert "directions=%d" % D in r.describe()


def test_calls_validate_arguments_before_any_device_work(lib):
    r = rnn.RNN(0, 1, 4, 2, 64, 64, 1)
    H = r.h
    assert lib.rnn_fwd(H, None, None, None, None, None, None, None, None, None, None) == -1
    assert lib.rnn_bwd_data(H, *([None] * 12)) == -1
    assert lib.rnn_bwd_weights(H, None, None, None, None, 0, None, None) == -1
    # misaligned pointer
    assert lib.rnn_fwd(H, ctypes.c_void_p(0x1001), None, None, ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000),
                       None, None, None, ctypes.c_void_p(0x4000), None) == -1
    assert lib.rnn_gemm_bf16(0, 1, 1, None, 8, 0, None, 8, 0, None, 1, None, 0, None) == -1
    assert lib.rnn_get_sizes(None, None, None, None, None) == -1


def test_persistent_plan_selection(lib):
    # small batch, supported width, one layer: persistent, no wavefront
    assert "recurrence=persistent" in rnn.RNN(0, 1, 10, 4, 64, 1024, 1).describe()
    assert "recurrence=streaming" in rnn.RNN(0, 2, 10, 4, 64, 1024, 1, flags=rnn.FLAG_FORCE_STREAMING).describe()
    assert "recurrence=persistent" not in rnn.RNN(0, 2, 10, 64, 64, 1024, 1).describe()
    with pytest.raises(rnn.RnnError) as e:
        rnn.RNN(0, 1, 10, 64, 64, 1024, 1, flags=rnn.FLAG_FORCE_PERSISTENT)
    assert e.value.code == -2
    with pytest.raises(rnn.RnnError):
        rnn.RNN(0, 1, 10, 4, 64, 1024, 0, flags=rnn.FLAG_FORCE_PERSISTENT)  # fp32 mode has no persistent path
    # widths the register-resident weights cover: LSTM and GRU up to 1024, simple RNNs up to 2048
    for cell, hmax in ((0, 1024), (1, 1024), (2, 2048), (3, 2048)):
        assert "recurrence=persistent" in rnn.RNN(cell, 1, 10, 8, 64, hmax, 1).describe()
        # wider: not persistent (the stacked forward where its chunks fit, else the step launches)
        assert "recurrence=persistent" not in rnn.RNN(cell, 1, 10, 8, 64, 2 * hmax, 1).describe()
        assert "recurrence=persistent" not in rnn.RNN(cell, 1, 10, 9, 64, hmax, 1).describe()
    # the hand-off variant the plan reports: clusters unless turned off
    d = rnn.RNN(0, 1, 10, 4, 64, 1024, 1).describe()
    assert "persist_cluster=0" not in d
    d = rnn.RNN(0, 1, 10, 4, 64, 1024, 1, flags=rnn.FLAG_NO_PERSIST_CLUSTER).describe()
    assert "persist_cluster=0" in d


def test_stacked_plan_groups(lib):
    """Persistent stacked forward (bf16, one direction, 9..64 sequences): the
    layers run in groups of up to 4 per launch, as many as fit on the SMs
    (layer 0: 32 units x K chunks of 512 per CTA over its recurrent part;
    higher layers also over their input part)."""
    import re

    def plan(*a, **k):
        d = rnn.RNN(*a, **k).describe()
        return re.search(r"recurrence=(\w+)", d).group(1), re.search(r"stack_groups=(\S+)", d).group(1)
    # 4-layer LSTM H=512 B=64: 16 + 3 x 32 CTAs, one launch
    assert plan(0, 4, 100, 64, 512, 512, 1) == ("stacked", "0+4")
    # 8-layer GRU H=1024 B=32: on 512-wide chunks layer 0 takes 64 CTAs and the
    # others 128 each; the higher layers of a pair widen to 1024-wide chunks
    # (64 CTAs; 896 k in TMEM, 128 in shared memory): two layers per launch
    assert plan(1, 8, 200, 32, 1024, 1024, 1) == ("stacked", "0+2,2+2,4+2,6+2")
    # B = 33..64 at H = 1024: the widened chunks do not fit shared memory, one layer per launch
    assert plan(1, 4, 100, 48, 1024, 1024, 1) == ("stacked", "0+1,1+1,2+1,3+1")
    # tanh H=1024 B=32: 8 + 16 + 16 + 16 + 16 CTAs -> 4 + 1
    assert plan(2, 5, 20, 32, 64, 1024, 1) == ("stacked", "0+4,4+1")
    # B <= 8: the single-layer persistent recurrence keeps the forward unless
    # forced or a stacked group holds several layers on chunks that fit TMEM
    assert plan(0, 1, 10, 4, 64, 1024, 1)[0] == "persistent"
    assert plan(0, 1, 10, 4, 64, 1024, 1, flags=rnn.FLAG_FORCE_STACK)[0] == "stacked"
    assert plan(0, 2, 10, 4, 64, 1024, 1)[0] == "persistent"  # two layers only on widened chunks
    assert plan(0, 2, 10, 4, 64, 1024, 1, flags=rnn.FLAG_FORCE_STACK) == ("stacked", "0+2")
    assert plan(0, 4, 100, 8, 512, 512, 1) == ("stacked", "0+4")
    # off: flag, streaming forced, wider batches, fp32, bidirectional, H not a multiple of 256
    assert plan(0, 4, 100, 64, 512, 512, 1, flags=rnn.FLAG_NO_STACK)[0] == "streaming"
    assert plan(0, 4, 100, 64, 512, 512, 1, flags=rnn.FLAG_FORCE_STREAMING)[0] == "streaming"
    assert plan(0, 4, 100, 65, 512, 512, 1)[0] == "streaming"
    assert plan(0, 4, 100, 32, 512, 512, 0)[0] == "streaming"
    assert plan(0, 2, 10, 32, 512, 512, 1, flags=rnn.FLAG_BIDIRECTIONAL)[0] == "streaming"
    assert plan(0, 2, 10, 32, 64, 320, 1)[0] == "streaming"
    with pytest.raises(rnn.RnnError):
        rnn.RNN(0, 2, 10, 32, 64, 320, 1, flags=rnn.FLAG_FORCE_STACK)
    # the backward, highest group first (host planning for GB300: clusters
    # of up to 8 CTAs, at most 152 CTAs per launch and 14 clusters of 8)
    bw = lambda *a, **k: re.search(r"stack_bwd_groups=(\S+)", rnn.RNN(*a, **k).describe()).group(1)
    assert bw(0, 4, 100, 64, 512, 512, 1) == "0+4"
    assert bw(2, 5, 8, 33, 96, 1024, 1) == "1+4,0+1"
    # GRU H=1024: a layer with the share from above (K = 2 G H = 6144, 768-wide
    # chunks) takes 64 CTAs, two of them 16 clusters of 8, which do not fit;
    # with each group's top layer on its recurrent product only ("r": 32
    # CTAs, the share from above computed by a GEMM) two layers per launch
    assert bw(1, 8, 200, 32, 1024, 1024, 1) == "6+2,4+2,2+2,0+2r"
    # LSTM H=1024: a lower layer's K = 8192 on 1024-wide chunks (896 k in TMEM,
    # 128 in shared memory: 64 CTAs) and a recurrent-only top (32 CTAs)
    assert bw(0, 4, 100, 32, 1024, 1024, 1) == "2+2,0+2r"
    # B = 33..64: two accumulators of 64 columns leave 768 k of TMEM; one layer per launch
    assert bw(0, 4, 100, 48, 1024, 1024, 1) == "3+1,2+1,1+1,0+1r"
    assert bw(0, 4, 100, 64, 512, 512, 1, flags=rnn.FLAG_NO_STACK_BWD) == "-"
    assert bw(0, 4, 100, 64, 512, 512, 1, flags=rnn.FLAG_NO_STACK) == "-"
    # variable lengths switch the forward to step launches
    r = rnn.RNN(0, 2, 10, 16, 64, 512, 1)
    assert "recurrence=stacked" in r.describe()
    r.set_lengths([10] * 8 + [5] * 8)
    assert "recurrence=streaming" in r.describe()
    r.set_lengths([10] * 16)
    assert "recurrence=stacked" in r.describe()


def test_wavefront_chunking_plan(lib):
    r = rnn.RNN(0, 4, 50, 256, 4096, 4096, 1, chunk=5)
    assert "chunk=5 nchunks=10" in r.describe()
    r = rnn.RNN(0, 4, 50, 256, 4096, 4096, 1, flags=rnn.FLAG_NO_WAVEFRONT)
    assert "wavefront=0 chunk=50 nchunks=1" in r.describe()


def test_backward_split_plan_invariants(lib):
    """Backward-step K splits: a power of two that the K blocks fill exactly
    (every split has work) and that cuts a tile into 16-column slices."""
    import re
    for cell in (0, 1, 2):
        G = {0: 4, 1: 3, 2: 1}[cell]
        for H in (64, 128, 192, 256, 320, 512, 768, 1024, 2048, 4096):
            for B in (1, 4, 32, 64, 130, 256):
                d = rnn.RNN(cell, 1, 3, B, 64, H, 1, flags=rnn.FLAG_FORCE_STREAMING).describe()
                bn = int(re.search(r"bwd_bn=(\d+)", d).group(1))
                sp = int(re.search(r"bwd_splits=(\d+)", d).group(1))
                kb = (G * H + 63) // 64
                per = -(-kb // sp)
                assert sp & (sp - 1) == 0 and -(-kb // per) == sp and bn % (16 * sp) == 0, (cell, H, B, bn, sp)


def test_transposed_step_plan(lib):
    """Recurrent steps taken as W_h h^T: chosen for many gate rows and at most
    256 batch entries (bf16 LSTM / tanh RNN), with packing unit 1; forced or
    refused by flags; every split count keeps the backward invariants."""
    import re
    d = rnn.RNN(0, 4, 50, 256, 4096, 4096, 1).describe()
    assert "transposed=1" in d and " u=1 " in d and "bwd_bn=256 bwd_splits=4" in d and "fused_point=1" in d
    assert "fused_point=0" in rnn.RNN(0, 4, 50, 256, 4096, 4096, 1, flags=rnn.FLAG_NO_FUSED_POINT).describe()
    assert "fused_point=0" in rnn.RNN(2, 1, 10, 256, 4096, 16384, 1).describe()  # tanh: separate kernel
    # several steps per launch: opt-in, LSTM, batch a multiple of 32, a step's tiles within the SM pairs
    assert "step_chunks=0" in d
    ch = lambda *a: rnn.RNN(*a, flags=rnn.FLAG_STEP_CHUNKS).describe()
    assert "step_chunks=1" in ch(0, 4, 50, 256, 4096, 4096, 1)
    assert "step_chunks=1" in ch(0, 2, 10, 96, 384, 384, 1)
    assert "step_chunks=0" in ch(0, 2, 10, 200, 2048, 2048, 1)   # 200 % 32
    assert "step_chunks=0" in ch(0, 2, 10, 256, 8192, 8192, 1)   # 128 tiles of 256 gate rows > 76 pairs
    assert "step_chunks=0" in ch(2, 2, 10, 256, 4096, 4096, 1)   # tanh
    d = rnn.RNN(0, 4, 50, 256, 4096, 4096, 1, flags=rnn.FLAG_NO_TRANSPOSED).describe()
    assert "transposed=0" in d and " u=64 " in d
    assert "transposed=0" in rnn.RNN(0, 4, 50, 257, 4096, 4096, 1).describe()   # batch wider than one tile
    assert "transposed=0" in rnn.RNN(1, 4, 50, 256, 4096, 4096, 1).describe()   # GRU keeps h W_h^T
    assert "transposed=1" in rnn.RNN(0, 2, 10, 64, 512, 512, 1).describe()      # measured faster there
    assert "transposed=0" in rnn.RNN(0, 2, 10, 256, 512, 512, 1).describe()     # ... but not at B=256
    assert "transposed=1" in rnn.RNN(0, 2, 10, 128, 256, 256, 1).describe()     # from H=256 at 64 <= B <= 128
    assert "transposed=0" in rnn.RNN(0, 2, 10, 32, 256, 256, 1).describe()
    assert "transposed=0" in rnn.RNN(0, 2, 10, 32, 1024, 1024, 1).describe()    # nor at H=1024, B<64
    assert "transposed=1" in rnn.RNN(0, 2, 10, 32, 2048, 2048, 1).describe()
    assert "transposed=1" in rnn.RNN(2, 2, 10, 16, 2048, 2048, 1).describe()    # tanh from H=2048
    assert "transposed=0" in rnn.RNN(2, 2, 10, 256, 1024, 1024, 1).describe()
    assert "transposed=1" in rnn.RNN(3, 2, 10, 64, 2048, 2048, 1).describe()    # ReLU RNN like tanh
    assert "recurrence=persistent" in rnn.RNN(3, 1, 10, 4, 64, 1024, 1).describe()
    for bad in [dict(cell=1, B=9, H=256, mode=1), dict(cell=0, B=300, H=256, mode=1), dict(cell=0, B=9, H=256, mode=0)]:
        with pytest.raises(rnn.RnnError):
            rnn.RNN(bad["cell"], 1, 3, bad["B"], 64, bad["H"], bad["mode"], flags=rnn.FLAG_FORCE_TRANSPOSED)
    for cell, G in ((0, 4), (2, 1)):
        for H in (64, 128, 192, 256, 512, 1024, 4096):
            for B in (1, 9, 64, 65, 129, 256):
                d = rnn.RNN(cell, 1, 3, B, 64, H, 1, flags=rnn.FLAG_FORCE_TRANSPOSED | rnn.FLAG_FORCE_STREAMING).describe()
                assert "transposed=1" in d and " u=1 " in d
                bn = int(re.search(r"bwd_bn=(\d+)", d).group(1))
                sp = int(re.search(r"bwd_splits=(\d+)", d).group(1))
                kb = (G * H + 63) // 64
                per = -(-kb // sp)
                assert bn >= min(256, B) and sp & (sp - 1) == 0 and -(-kb // per) == sp and bn % (16 * sp) == 0 \
                    and sp <= 8, (cell, H, B, bn, sp)


def test_set_lengths_validation_and_plan(lib):
    """Lengths must be 1..T and non-increasing; a handle planned with the
    persistent recurrence switches to step launches once lengths differ."""
    r = rnn.RNN(0, 1, 10, 4, 64, 1024, 1)
    assert "recurrence=persistent" in r.describe()
    with pytest.raises(ValueError):
        r.set_lengths([10, 9, 8])
    for bad in ([10, 11, 3, 1], [0, 0, 0, 0], [3, 5, 5, 1]):
        with pytest.raises(rnn.RnnError) as e:
            r.set_lengths(bad)
        assert e.value.code == -1
    assert "recurrence=persistent" in r.describe()
    r.set_lengths([10, 10, 10, 10])            # all full: nothing changes
    assert "recurrence=persistent" in r.describe()
    r.set_lengths([10, 7, 7, 2])
    assert "recurrence=streaming" in r.describe()
    r.set_lengths(None)
    assert "recurrence=persistent" in r.describe()


def test_bidirectional_plan_and_sizes(lib):
    """Bidirectional stacks: two weight sets per layer (the next layer's input
    is 2H wide), states per (layer, direction), no wavefront; small bf16
    batches take the persistent recurrence (one launch per direction) unless
    lengths differ."""
    import oracle
    for cell, mode in ((0, 1), (1, 1), (2, 0), (3, 1)):
        L, T, B, I, H = 3, 10, 4, 64, 128
        r = rnn.RNN(cell, L, T, B, I, H, mode, flags=rnn.FLAG_BIDIRECTIONAL)
        d = r.describe()
        assert "directions=2" in d and "wavefront=0" in d
        assert ("recurrence=persistent" if mode == 1 else "recurrence=streaming") in d
        e = 2 if mode == 1 else 4
        assert r.sizes()["user_weights"] == oracle.weight_count(cell, L, I, H, D=2) * e
        uni = rnn.RNN(cell, L, T, B, I, H, mode)
        assert "directions=1" in uni.describe()
        assert r.sizes()["reserve"] > uni.sizes()["reserve"]
    r = rnn.RNN(0, 1, 10, 4, 64, 1024, 1, flags=rnn.FLAG_BIDIRECTIONAL)
    assert "recurrence=persistent" in r.describe()
    r.set_lengths([10, 7, 7, 2])
    assert "recurrence=streaming" in r.describe()
    r.set_lengths(None)
    assert "recurrence=persistent" in r.describe()
    rb = rnn.RNN(0, 1, 10, 64, 64, 1024, 1, flags=rnn.FLAG_BIDIRECTIONAL)
    assert "recurrence=streaming" in rb.describe()


@pytest.mark.parametrize("wl", [synth.WORKLOADS[1], synth.WORKLOADS[5], synth.WORKLOADS[6],
                                synth.Workload("g", 1, 2, 3, 4, 8, 16, 0, state_std=0.3, directions=2)],
                         ids=lambda w: w.name)
def test_device_generator_matches_host_generator(wl):
    """The inputs the benchmark draws on the device (here on the CPU) are the
    host arrays the parity tests use: the same counters per tensor, per layer
    and per direction (normals may differ in the last float32 ulp)."""
    import numpy as np
    import torch
    small = wl.replace(T=min(wl.T, 3), B=min(wl.B, 4), hidden=min(wl.hidden, 64), input=min(wl.input, 64))
    w_dev = synth.device_tensor(small, "w", "cpu", torch.float32).numpy().astype(np.float64)
    w_host = synth.flat_weights(small).astype(np.float32).astype(np.float64)
    assert w_dev.shape == w_host.shape == (small.weight_count(),)
    np.testing.assert_array_equal(w_dev, w_host)
    for what, host in (("x", synth.make_x(small)), ("dy", synth.make_dy(small)), ("h0", synth.make_state(small, "h0"))):
        dev = synth.device_tensor(small, what, "cpu", torch.float32).numpy().astype(np.float64)
        assert dev.shape == host.shape, what
        np.testing.assert_allclose(dev, host.astype(np.float32), rtol=1e-6, atol=1e-6, err_msg=what)


def test_fp8_stash_plan_and_sizes(lib):
    """RNN_FLAG_FP8_STASH: bf16 persistent inference with e4m3 W_h up to H=2048
    (LSTM, GRU); the packed buffer gains G*H*H bytes and G*H scales per layer;
    refused where no persistent plan exists or in the fp32 mode."""
    for cell, H, B in [(0, 2048, 4), (1, 2048, 8), (0, 256, 3), (2, 1024, 5)]:
        a = rnn.RNN(cell, 2, 8, B, 64, H, 1, flags=rnn.FLAG_FP8_STASH)
        b = rnn.RNN(cell, 2, 8, B, 64, H, 1)
        assert "fp8_stash=1" in a.describe() and "fp8_stash=0" in b.describe()
        G = synth.GATES[cell]
        extra = a.sizes()["packed_weights"] - b.sizes()["packed_weights"]
        assert extra >= 2 * (G * H * H + G * H * 4) and extra <= 2 * (G * H * H + G * H * 4) + 4 * 256
        assert a.sizes()["workspace"] >= b.sizes()["workspace"]
    for bad in [dict(mode=0, hidden=256), dict(B=16, hidden=256), dict(hidden=4096), dict(flags_extra=rnn.FLAG_FORCE_STREAMING)]:
        kw = dict(cell=0, layers=1, T=4, B=4, input=64, hidden=512, mode=1)
        extra = bad.pop("flags_extra", 0)
        kw.update(bad)
        with pytest.raises(rnn.RnnError) as e:
            rnn.RNN(**kw, flags=rnn.FLAG_FP8_STASH | extra)
        assert e.value.code == -2
