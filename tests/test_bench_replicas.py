"""bench.py with N > 1 runs independent replicas and reports the slowest
rank's time: its process-group set-up, max-over-ranks reduction and barrier
are checked here with two gloo ranks on the CPU (no GPU involved)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    ws, r, local = bench.dist_init()
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(ws)
    # rank r reports a step time of r + 1.5 ms; every rank must see the max
    got = bench.reduce_max(rank + 1.5, ws)
    import torch.distributed as dist
    dist.destroy_process_group()
    out.put((rank, got))


def test_two_gloo_replicas_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 2.5, 1: 2.5}


def test_single_process_needs_no_process_group():
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25
