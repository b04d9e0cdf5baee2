"""The benchmark's multi-rank host logic on CPU: two gloo ranks on
127.0.0.1. Each rank is an independent replica; the only cross-rank steps
are the barrier and the max over ranks of the timings, and only rank 0
prints the reference arm's line."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d, r, w, local = bench._dist()
    assert (r, w, local) == (rank, world, rank) and d is dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench._reduce_max(dist, [1.0 + rank, 10.0 - rank], "cpu")
    # the ranks agree on skipping the end-to-end step when any one cannot run it
    agree = (bench._all_ranks(dist, True, "cpu"), bench._all_ranks(dist, rank == 0, "cpu"))
    assert agree == (True, False), agree
    dist.barrier()
    dist.destroy_process_group()
    # the reference arm: every rank but 0 exits at once without work or output
    buf = io.StringIO()
    if rank != 0:
        args = type("A", (), {"config": 1, "steps": 1, "warmup": 1, "gpus": world})()
        with redirect_stdout(buf):
            bench.run_reference(args)
    out.put((rank, got, buf.getvalue()))


@pytest.mark.timeout(300)
def test_two_gloo_ranks_reduce_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, q), nprocs=2, start_method="spawn", join=True)
    res = sorted(q.get() for _ in range(2))
    for rank, got, printed in res:
        assert got == [2.0, 10.0]
        if rank != 0:
            assert printed == ""


def test_single_process_has_no_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    sys.path.insert(0, ROOT)
    import bench
    assert bench._dist() == (None, 0, 1, 0)
    assert bench._all_ranks(None, True, "cpu") and not bench._all_ranks(None, False, "cpu")
