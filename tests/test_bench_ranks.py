"""The replicas path of the benchmark on CPU: two gloo ranks (one process each,
127.0.0.1) take each timing's maximum over the ranks, which is what the bench
line reports under torchrun; a single process keeps its own values."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_sync()
        got = bench.slowest_rank([1.0 + rank, 10.0 - rank, 0.5], torch.device("cpu"))
        bench.rank_sync()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = dict(q.get(timeout=120) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    assert res[0] == res[1] == [2.0, 10.0, 0.5]


def test_single_process_keeps_its_values():
    assert bench.slowest_rank([3.0, 4.0], torch.device("cpu")) == [3.0, 4.0]
    bench.rank_sync()
