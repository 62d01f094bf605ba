"""The bench's multi-process path on the CPU: two gloo ranks. The replicas exchange nothing but
a barrier and the max of their times, and the reported value is the units of all ranks over
the slowest rank's time. The reference arm does its work on rank 0 only."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    slowest = bench._max_over_ranks(10.0 * (rank + 1), ws)   # rank times 10 ms and 20 ms
    bench._barrier(ws)
    rate = bench._job_rate(1000, slowest, ws)                 # 1000 units per rank
    q.put((rank, slowest, rate))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_job_rate():
    pytest.importorskip("torch")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, rate in out:
        assert slowest == 20.0                      # the max over ranks, on every rank
        assert abs(rate - 2 * 1000 / 0.020) < 1e-6  # all units over the slowest time


def _ref_worker(rank, ws, port, q):
    # the reference arm under torchrun: rank 0 alone runs and prints; the others exit with 0
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import io
    import contextlib
    import types
    import bench
    buf = io.StringIO()
    args = types.SimpleNamespace(steps=1, warmup=0, gpus=ws)
    with contextlib.redirect_stdout(buf):
        bench.bench_reference(args)
    q.put((rank, buf.getvalue()))


def test_reference_arm_runs_on_rank_zero_only():
    pytest.importorskip("torch")
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ref_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=600) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[1] == ""
    assert '"impl": "reference"' in out[0]
