"""bench.py's rank helpers on CPU: two gloo ranks on 127.0.0.1.

The benchmark runs one replica per GPU (the shape-fused update exchanges
nothing between members, so the path has no collective); the ranks only meet
in a barrier around the timed region and in a max over their step times.
"""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": "2",
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    world, r, local = bench.dist_setup()
    bench.barrier(world)
    m = bench.allmax(world, 10.0 + 5.0 * r)  # rank 1 is the slower one
    bench.barrier(world)
    q.put((r, world, local, m))
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2, 0, 15.0), (1, 2, 1, 15.0)]


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.allmax(1, 3.5) == 3.5
    bench.barrier(1)
