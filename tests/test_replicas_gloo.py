"""The N>1 path of bench.py (independent replicas, one per GPU) on CPU: two
gloo ranks exercise the host-side reductions it uses -- max of the step time
over ranks, mean of the share over ranks, and the barrier."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "C3_DIST_BACKEND": "gloo"})
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse_args([])
    world_, rank_, local_, pg = bench.dist_init(args)
    try:
        step_ms = 10.0 + 5.0 * rank          # ranks differ: the slower one sets the step time
        share = 40.0 + 20.0 * rank
        bench.barrier(pg)
        got_max = bench.reduce_max(pg, step_ms)
        got_mean = bench.reduce_mean(pg, share)
        bench.barrier(pg)
        q.put((rank_, world_, got_max, got_mean))
    finally:
        pg.destroy_process_group()


def test_two_gloo_ranks_reduce_like_bench():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = sorted(q.get(timeout=10) for _ in range(world))
    for rank, w, got_max, got_mean in results:
        assert w == world
        assert got_max == 15.0
        assert got_mean == 50.0


def test_single_process_reductions_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(None, 3.5) == 3.5
    assert bench.reduce_mean(None, 7.0) == 7.0
    bench.barrier(None)
