"""The multi-rank host logic of bench.py on CPU with the gloo backend
(world size 2, 127.0.0.1): every rank gets its own input sets, the job time
is the slowest rank's (MAX all-reduce), the job throughput counts every
rank's units, and the reference arm runs on rank 0 only."""
import io
import os
import sys
import contextlib

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(1.5 + rank, dist, torch.device("cpu"))
        sets = [bench.rank_set_index(rank, s) for s in range(3)]
        gathered = [None] * world
        dist.all_gather_object(gathered, sets)
        # the reference arm prints on rank 0 only; other ranks return without work
        buf = io.StringIO()
        args = type("A", (), dict(workload="c1", ref_requests=1, warmup=0, steps=1))()
        with contextlib.redirect_stdout(buf):
            bench.run_reference(args)
        q.put((rank, t, gathered, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    import socket
    with socket.socket() as s_:
        s_.bind(("127.0.0.1", 0))
        port = s_.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    for rank, t, gathered, printed in out:
        assert t == 2.5                                    # the slowest rank's time
        assert not set(gathered[0]) & set(gathered[1])     # disjoint input sets
        assert (printed.strip() != "") == (rank == 0)      # rank 0 alone reports
    import bench
    assert bench.job_throughput(1024, 2, 10, 20.0) == pytest.approx(1024 * 2 * 10 / 0.02)
