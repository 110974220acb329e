"""The multi-process (replica) path of bench.py on CPU with the gloo backend: rank set-up
from the torchrun environment, the barrier, the max-reduction of per-rank timings and
the whole-job aggregate.  Two ranks, 127.0.0.1 rendezvous."""
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
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "MSA_BENCH_BACKEND": "gloo"})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, loc = bench.dist_setup()
    bench.barrier(w)
    times = bench.reduce_max([1.0 + rank, 5.0 - rank], w)
    agg = bench.aggregate([10.0] * w, times[0])
    q.put((r, w, loc, times, agg))
    dist.destroy_process_group()


def test_two_rank_reduction_and_aggregate():
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
    for (r, w, loc, times, agg) in res:
        assert w == 2 and loc == r
        assert times == [2.0, 5.0]          # element-wise max over ranks
        assert agg == pytest.approx(20.0 / 2.0)


def test_reference_arm_other_ranks_do_nothing():
    sys.path.insert(0, ROOT)
    import bench

    class A:
        pass
    assert bench.run_reference(A(), 2, 1) is None
