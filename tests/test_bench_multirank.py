"""Host-side logic of the multi-GPU benchmark run, on CPU with two gloo
ranks: the timing is the maximum over ranks, the throughput counts every
rank's rows, and the reference arm prints from rank 0 only."""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        value = bench.job_throughput(512, world, ms, 100)
        os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
        buf = io.StringIO()
        if rank != 0:
            with contextlib.redirect_stdout(buf):
                bench.reference_arm(None)
        q.put((rank, ms, value, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_and_count_every_row():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value, out in res:
        assert ms == 15.0                        # the slower rank's time, on both ranks
        assert value == pytest.approx(2 * 512 / (15.0 / 1e3 / 100))
        if rank != 0:
            assert out == ""                     # non-zero ranks print nothing


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(512, 1, 1000.0, 1000) == pytest.approx(512000.0)
