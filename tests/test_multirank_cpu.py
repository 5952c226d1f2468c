"""The N > 1 path of the benchmark on CPU: world-size-2 gloo ranks run
independent replicas; the step time is the maximum over ranks and the value
is the whole-job aggregate.  No GPU and no collective on the data path."""
import os
import socket
import sys

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


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = 10.0 + 5.0 * rank          # rank 1 is the slow replica
    ms, tflops, w = bench.replica_aggregate(ms_local, 2.0e12, dist, "cpu")
    dist.barrier()
    out[rank] = (ms, tflops, w)
    dist.destroy_process_group()


def test_replicas_take_max_time_and_aggregate_work():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms, tflops, w = res[r]
        assert w == 2
        assert ms == pytest.approx(15.0)                        # max over ranks
        assert tflops == pytest.approx(2 * 2.0e12 / 15e-3 / 1e12)  # both replicas' work over the slowest time


def test_single_process_aggregate():
    sys.path.insert(0, ROOT)
    import bench
    ms, tflops, w = bench.replica_aggregate(20.0, 4.0e12)
    assert (ms, w) == (20.0, 1) and tflops == pytest.approx(200.0)


def test_reference_arm_prints_one_contract_line():
    """bench.py --impl reference times the oracle on the host and prints the
    benchmark's JSON line with impl, e2e and cpu_baseline (no GPU involved)."""
    import json
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--config", "0",
                          "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["steps"] == 1 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert "columns" in d["cpu_baseline"]["sample"]
