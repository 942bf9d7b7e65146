"""Replica (N>1) host logic of the benchmark on two gloo ranks on the CPU:
the whole-job time is the slowest rank's, the routed tokens are summed, and
every rank draws its own batch.  No GPU and no data-path collective: the
method partitions into independent batches, one per GPU."""
import os

import pytest
import torch.multiprocessing as mp


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mx, sm = bench.reduce_across_ranks([1.5 + rank, 10.0 * (rank + 1)], [100 + rank], dist, "cpu")
    out[rank] = (mx, sm, bench.rank_seed(rank, 3))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        mx, sm, seed = out[r]
        assert mx == [2.5, 20.0]          # slowest rank's times
        assert sm == [201.0]              # tokens of both replicas
    assert out[0][2] != out[1][2]         # disjoint batches per replica


def test_single_process_is_identity():
    import bench
    assert bench.reduce_across_ranks([3.0], [7], None) == ([3.0], [7])
