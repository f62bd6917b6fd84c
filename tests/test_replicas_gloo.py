"""The multi-rank path of bench.py (independent replicas, max-over-ranks
timing) with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [1.0 + rank, 10.0 - rank]  # rank 1 slower on the first, rank 0 on the second
    got = bench.max_over_ranks(ms, world)
    thr = bench.replica_throughput(32, world, got[0])
    seed = bench.replica_seed(rank)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got, thr, seed))


def test_two_rank_replica_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, thr, seed in res:
        assert got == [2.0, 10.0]
        assert thr == pytest.approx(32 * 2 / 2.0e-3)
    assert res[0][3] != res[1][3]  # independent replicas
