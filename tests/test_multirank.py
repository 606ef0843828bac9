"""The benchmark's multi-rank aggregation on CPU (gloo, world size 2): each
rank times its own replica of the workload; the job's time is the max over
ranks and its work the sum (replicas, weak scaling, no data-path
collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (rank, world, rank)
    elapsed = [0.25, 0.40][rank]
    units = [1000.0, 3000.0][rank]
    t, u = bench.aggregate(elapsed, units, world)
    out.put((rank, t, u))
    dist.destroy_process_group()


def test_aggregate_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, u in res:
        assert t == pytest.approx(0.40)
        assert u == pytest.approx(4000.0)


def test_aggregate_single_rank_is_identity():
    import bench
    assert bench.aggregate(1.5, 7.0, 1) == (1.5, 7.0)
