"""Data-parallel training over batch shards with world-size-2 gloo ranks on
CPU, through the same helpers the benchmark's data-parallel step uses
(recurrent_neural_network_gb300.dp): each rank takes its shard of the global
batch with dp.shard, runs the double-precision oracle on it, and sums its
weight gradients with dp.allreduce_grads_.  The result must equal the
full-batch weight gradient (sequences are independent, so dW is a sum over
batch entries), while each rank's dx, dh0, dc0 are the full-batch values of
its own columns.  This is the one exchange step a data-parallel training step
adds to the path; no GPU is involved."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _inputs(cell, directions=1):
    from recurrent_neural_network_gb300 import runner, synth
    wl = synth.Workload(name="dp", cell=cell, layers=2, T=4, B=6, input=5, hidden=4, mode=synth.MODE_FP32,
                        forget_bias=1.0, state_std=0.3, kink_margin=0.75 if cell == 3 else 0.0,
                        directions=directions)
    return wl, runner.HostInputs(wl, with_state_grads=True)


def _bwd(hi):
    import oracle
    w = hi.wl
    return oracle.bwd(w.cell, w.layers, w.T, w.B, w.input, w.hidden, hi.x, hi.w, hi.dy, h0=hi.h0, c0=hi.c0,
                      dhT=hi.dhT, dcT=hi.dcT, D=w.directions)


def _rank(rank, world, port, cell, directions, out):
    sys.path.insert(0, ROOT)
    from recurrent_neural_network_gb300 import dp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl, hi = _inputs(cell, directions)
    # this rank's shard of every batch-indexed input, as torch tensors (the benchmark's form)
    sh = object.__new__(type(hi))
    sh.wl = wl.replace(B=wl.B // world)
    sh.w = hi.w
    for k in ("x", "h0", "c0", "dy", "dhT", "dcT"):
        a = getattr(hi, k)
        t = None if a is None else dp.shard(torch.from_numpy(a), rank, world, dim=1)
        setattr(sh, k, None if t is None else t.numpy())
    dx, dh0, dc0, dw = _bwd(sh)
    t = torch.from_numpy(np.ascontiguousarray(dw))
    assert dp.allreduce_grads_(t) is t
    k = wl.B // world
    out[rank] = (list(range(rank * k, (rank + 1) * k)), dx, dh0, dc0, t.numpy().copy())
    dist.destroy_process_group()


@pytest.mark.parametrize("cell,directions", [(0, 1), (1, 1), (2, 1), (3, 1), (0, 2)],
                         ids=["lstm", "gru", "tanh", "relu", "lstm_bidir"])
def test_batch_shards_plus_allreduce_equal_full_batch(cell, directions):
    sys.path.insert(0, ROOT)
    import oracle
    oracle.build()
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, cell, directions, out), nprocs=world, join=True)
        res = dict(out)
    wl, hi = _inputs(cell, directions)
    dx, dh0, dc0, dw = _bwd(hi)
    for r in range(world):
        cols, rdx, rdh0, rdc0, rdw = res[r]
        np.testing.assert_allclose(rdw, dw, rtol=1e-12, atol=1e-14 * np.abs(dw).max())
        np.testing.assert_allclose(rdx, dx[:, cols], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(rdh0, dh0[:, cols], rtol=1e-12, atol=1e-15)
        if dc0 is not None:
            np.testing.assert_allclose(rdc0, dc0[:, cols], rtol=1e-12, atol=1e-15)


def test_shard_and_global_batch_helpers():
    sys.path.insert(0, ROOT)
    from recurrent_neural_network_gb300 import dp, synth
    wl = synth.WORKLOADS[3]
    g = dp.global_batch(wl, 4)
    assert g.B == 4 * wl.B and g.T == wl.T and g.hidden == wl.hidden
    assert dp.global_batch(wl, 1) == wl
    a = np.arange(2 * 8 * 3).reshape(2, 8, 3)
    parts = [dp.shard(a, r, 4) for r in range(4)]
    np.testing.assert_array_equal(np.concatenate(parts, axis=1), a)
    t = torch.from_numpy(a)
    assert torch.equal(dp.shard(t, 1, 4), t[:, 2:4])
    assert dp.shard(None, 0, 2) is None
    with pytest.raises(ValueError):
        dp.shard(a, 0, 3)
    x = torch.ones(3)
    assert dp.allreduce_grads_(x) is x and torch.equal(x, torch.ones(3))  # no process group: no-op
