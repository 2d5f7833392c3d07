"""Multi-rank host logic of bench.py on CPU with the gloo backend (world size 2): the
max-over-ranks reduction and the whole-job throughput (all ranks' units over the slowest
rank's time).  The data path has no collective; ranks are independent replicas."""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        # rank r took (r + 1) seconds for the same 10 units: throughput = 20 / 2
        thr = bench.aggregate(10.0, float(rank + 1), world)
        mx = bench.reduce_max([float(rank), 5.0 - rank, 3.0])
        bench.barrier()
        out.put((rank, thr, mx))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, thr, mx in res:
        assert thr == pytest.approx(10.0)
        assert mx == [1.0, 5.0, 3.0]


def test_single_process_is_identity():
    import bench

    assert bench.reduce_max([1.5, 2.5]) == [1.5, 2.5]
    assert bench.aggregate(8.0, 2.0, 1) == 4.0
