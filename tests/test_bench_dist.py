"""The benchmark's multi-rank plumbing on CPU: two gloo ranks, barrier, max
over ranks and the whole-job aggregate (bytes of all ranks over the slowest
rank's time)."""
import os
import socket
import sys

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
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, l = bench.dist_env()
    assert (w, r, l) == (world, rank, rank)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    t = 1.0 + rank          # rank 1 is the slower one
    agg = bench.aggregate(100.0, t, w)
    mx = bench.allreduce_max(float(rank * 10), w)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((rank, agg, mx))


def test_two_gloo_ranks_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, agg, mx in res:
        assert agg == pytest.approx(200.0 / 2.0)     # 2 ranks x 100 bytes over max time 2 s
        assert mx == 10.0


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(100.0, 4.0, 1) == 25.0
    assert bench.allreduce_max(3.0, 1) == 3.0
