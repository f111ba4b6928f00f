"""The multi-process path of the benchmark on CPU (gloo, world size 2): every
rank times its own replica of the step, the job time is the maximum over
ranks, and only rank 0 reports; the reference arm runs on rank 0 alone."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        mine = [1.0 + rank, 10.0 - rank]                   # rank-dependent step and e2e times
        got = bench.max_over_ranks(dist, mine, device="cpu")
        # the reference arm prints nothing on ranks other than 0
        out = io.StringIO()
        if rank != 0:
            class A:
                steps, warmup = 1, 0
            with redirect_stdout(out):
                bench.run_reference(A())
        dist.barrier()
        q.put((rank, got, out.getvalue()))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_rank0_reporting_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        rank, got, out = q.get(timeout=120)
        res[rank] = (got, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        assert res[rank][0] == [2.0, 10.0]           # max over ranks, element-wise
    assert res[1][1] == ""                            # rank 1 stays silent


def test_single_process_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, [3.0, 4.0]) == [3.0, 4.0]
