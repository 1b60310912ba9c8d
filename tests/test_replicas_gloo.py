"""Multi-process host logic of bench.py (N > 1 replicas) on CPU with gloo, world size 2.

Each rank times its own replica; the job time is the max over ranks and the
throughput counts the elements of every rank.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = [120.0, 150.0][rank]
    ms, value = bench.combine_ranks(ms_local, 1000 * 10**6, world, torch.device("cpu"))
    q.put((rank, ms, value))
    dist.destroy_process_group()


def test_combine_ranks_gloo():
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
    for rank, ms, value in res:
        assert ms == 150.0                       # max over ranks
        assert value == pytest.approx(2 * 1000e6 / 0.150 / 1e9)  # both ranks' elements


def test_combine_ranks_single():
    import bench
    ms, value = bench.combine_ranks(10.0, 10**9, 1, None)
    assert ms == 10.0 and value == pytest.approx(100.0)
