"""The N > 1 path of the benchmark on CPU: replicas over gloo, world size 2.

The convolution shards into independent images with no exchange, so `bench.py --gpus N` runs N
independent replicas; the only collectives are the timing barrier and the max of the measured
times over ranks.  These tests run that host logic in two processes over gloo (no GPU), plus the
reference arm's rule that only rank 0 works and prints.
"""
import contextlib
import io
import multiprocessing as mp
import os
import socket
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        step_ms = 10.0 * (rank + 1)          # rank 1 is the slow replica
        slowest = bench.max_over_ranks(step_ms, world, "cpu")
        value = bench.whole_job_tflops(world, 2.0e12, 5, slowest)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_replica_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    # both ranks see the slower replica's 20 ms; the job did 2 replicas x 5 steps x 2 TFLOP
    assert [g[1] for g in got] == [20.0, 20.0]
    assert all(abs(g[2] - 2 * 2.0e12 * 5 / 20e-3 / 1e12) < 1e-9 for g in got)


def test_one_rank_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, 1, "cpu") == 7.5
    assert bench.whole_job_tflops(1, 1.0e12, 4, 2.0) == pytest.approx(2000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    """Under torchrun the CPU reference arm works and prints on rank 0; other ranks exit at once."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    out = io.StringIO()
    args = types.SimpleNamespace(steps=1, warmup=0, gpus=2)
    with contextlib.redirect_stdout(out):
        assert bench.reference_arm(args) is None
    assert out.getvalue() == ""
