"""The benchmark's multi-GPU logic, run as two gloo ranks on the CPU.

Every rank runs its own copy of the workload (independent problems, no
collective on the data path); the only cross-rank step is the max over ranks
of the step time, and the whole-job value counts all ranks' FLOPs.  The
reference arm prints from rank 0 only; other ranks exit without work.
"""
import os
import socket
import sys
from pathlib import Path

import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parent.parent


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, str(ROOT))
    import bench
    w, r, local, dist = bench.dist_setup(backend="gloo")
    try:
        my_ms = 2.0 + rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(my_ms, dist)
        value = bench.whole_job_value(4.0e12, w, slowest)
        out[rank] = (w, r, slowest, value)
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert set(res) == {0, 1}
    for r in range(world):
        w, rr, slowest, value = res[r]
        assert w == 2 and rr == r
        assert slowest == 3.0  # max over ranks
        assert value == pytest.approx(2 * 4.0e12 / 3.0e-3 / 1e12)  # all ranks' work / slowest time


def _ref_rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, str(ROOT))
    import contextlib
    import io

    import bench

    class Args:
        steps, warmup, gpus = 1, 0, world
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(Args, bench.get_workload("tiny_nc"))
    q.put((rank, buf.getvalue()))


def test_reference_arm_prints_nothing_on_other_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_ref_rank, args=(1, 2, _free_port(), q))
    p.start()
    p.join(timeout=120)
    assert p.exitcode == 0
    rank, text = q.get(timeout=10)
    assert rank == 1 and text == ""
