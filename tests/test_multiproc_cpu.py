"""Multi-process rank arithmetic of bench.py on CPU (gloo, world size 2).

The hot path partitions into independent problems, so N GPUs run N replicas of
the per-GPU workload with no data-path collective; the only cross-rank steps are
the barrier and the reductions that turn per-rank times and units into the
whole-job figure.  These run here as two gloo processes.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        # rank r processed 100·(r+1) units in (r+1) seconds
        units, secs = 100.0 * (r + 1), float(r + 1)
        bench.barrier(w)
        agg = bench.aggregate_throughput(units, secs, w)
        mx = bench.max_over_ranks(secs, w)
        sm = bench.sum_over_ranks(units, w)
        q.put((r, w, local, agg, mx, sm))
    finally:
        dist.destroy_process_group()


def test_rank_reductions_world_size_two():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[0] for o in out] == [0, 1] and all(o[1] == 2 for o in out)
    for r, w, local, agg, mx, sm in out:
        assert local == r
        assert mx == pytest.approx(2.0)            # slowest rank's time
        assert sm == pytest.approx(300.0)          # all units of all ranks
        assert agg == pytest.approx(300.0 / 2.0)   # whole-job throughput


def test_single_process_reductions_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.sum_over_ranks(7.0, 1) == 7.0
    assert bench.aggregate_throughput(10.0, 2.0, 1) == pytest.approx(5.0)
