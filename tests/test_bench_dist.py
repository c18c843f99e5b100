"""The multi-rank host logic of bench.py (replicas: rendezvous, barrier,
max-over-ranks timing) on two CPU processes with the gloo backend."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    w, r, local = bench.init_dist()
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.5 + r, w)       # per-rank ms/step
    tokens = 1000
    value = tokens * w / (slowest * 1e-3)             # whole-job throughput
    q.put((r, w, slowest, value))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_rank_replicas_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(world))
    for r, w, slowest, value in res:
        assert w == 2 and slowest == pytest.approx(2.5)
        assert value == pytest.approx(1000 * 2 / 2.5e-3)
