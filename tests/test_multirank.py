"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each a
replica with its own timing; the reported time is the max over ranks and the
throughput is the aggregate of both replicas.  No GPU."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r's replica took (r + 1) ms for its step and 10*(r + 1) ms end to end
    got = bench.max_over_ranks([1.0 * (rank + 1), 10.0 * (rank + 1)], dist)
    gbs = bench.aggregate_gbs(1e9, got[0] * 1e-3, world)
    q.put((rank, got, gbs))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, got, gbs in res:
        assert got == [2.0, 20.0]                 # the slowest replica's times
        assert abs(gbs - 2 * 1e9 / 2e-3 / 1e9) < 1e-9   # 2 replicas x 1 GB in 2 ms


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.aggregate_gbs(2e9, 1.0, 1) == 2.0
