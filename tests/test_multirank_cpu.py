"""The multi-rank path of bench.py on CPU: two gloo ranks.

The pairs are independent, so N GPUs run N replicas with no collective on the
data path; what N > 1 adds is host logic: the process group, the barrier
around the timed region, the maximum of the ranks' times and the whole-job
value, and the reference arm printing on rank 0 alone.  These tests run that
logic as two spawned CPU processes over gloo (127.0.0.1).
"""
from __future__ import annotations

import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    r, local, w, dist = bench.dist_setup(world)
    assert (r, local, w) == (rank, rank, world) and dist is not None
    bench.barrier(dist)
    # each rank "timed" a different duration; the job is as slow as its slowest rank
    ms = bench.max_over_ranks(10.0 * (rank + 1), dist, "cpu")
    value = bench.job_value(1000, w, ms)
    # the reference arm prints on rank 0 only
    buf = io.StringIO()

    class Args:
        gpus, steps, warmup = world, 1, 0
    if rank != 0:
        with redirect_stdout(buf):
            bench.run_reference(Args, None)   # returns before touching the workload
    bench.barrier(dist)
    dist.destroy_process_group()
    out.put((rank, ms, value, buf.getvalue()))


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_value():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0, f"rank process exited with {p.exitcode}"
    res = sorted(out.get() for _ in range(world))
    for rank, ms, value, printed in res:
        assert ms == pytest.approx(20.0)                # max over ranks, seen by both
        assert value == pytest.approx(1000 * 2 / 0.020)  # units of all ranks over the slowest time
        assert printed == ""                             # only rank 0 prints the reference line


def test_single_process_skips_the_process_group(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup(1) == (0, 0, 1, None)
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
