"""The N > 1 path of the benchmark on CPU: two gloo ranks (127.0.0.1) run the
benchmark's barrier and max-over-ranks timing, and the whole-job figure is
the per-rank throughput times the replicas at the slowest rank's time.  The
hot path itself has no exchange step (replicas only), so no collective of the
library is involved."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(True)
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slower replica
        out[rank] = bench.max_over_ranks(local_ms, True)
        bench.barrier(True)
    finally:
        torch.distributed.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        assert dict(out) == {0: 15.0, 1: 15.0}
    sys.path.insert(0, ROOT)
    import bench
    # 1000 calls of 75.5 MB in 25 ms per step on each of 2 replicas
    assert bench.aggregate_gbps(1000, 75_513_864, 25.0, 2) == pytest.approx(2 * 3020.55, rel=1e-4)
    assert bench.max_over_ranks(7.0, False) == 7.0
