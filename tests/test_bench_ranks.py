"""The bench's multi-rank path on the CPU: two gloo ranks, as torchrun would launch them.

Each rank is an independent replica; the job's time is the slowest rank's (a max-reduction),
the whole-job throughput counts every rank's tokens, and the reference arm runs on rank 0
only (the other ranks return without work)."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slow = bench.ranks_max([1.5, 4.25][rank], "cpu")  # rank 1 is the slow one
        fast = bench.ranks_max([-3.0, -7.0][rank], "cpu")
        buf = io.StringIO()
        with redirect_stdout(buf):
            bench.run_reference(None, None, rank) if rank != 0 else None
        out.put((rank, slow, fast, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_only_rank0_reports():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [4.25, 4.25]
    assert [g[2] for g in got] == [-3.0, -3.0]
    assert got[1][3] == ""  # the reference arm prints nothing on rank 1


def test_single_process_needs_no_group_and_throughput_counts_every_rank():
    import bench

    assert bench.ranks_max(2.5, "cpu") == 2.5
    # 8 tokens per step, 100 steps in 2 s on each of 4 replicas
    assert bench.whole_job_tok_s(8, 100, 2.0, 4) == pytest.approx(1600.0)
    assert bench.whole_job_tok_s(1, 50, 0.125, 1) == pytest.approx(400.0)
