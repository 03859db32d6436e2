"""bench.py's multi-process plumbing on CPU: two gloo ranks, barrier, max and sum over ranks
(the only collectives the bench uses; the verify path itself shards with no exchange)."""

import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    try:
        d.barrier()
        q.put((rank, d.world, d.max(1.5 + rank), d.sum(10.0 * (rank + 1)),
               d.pg.get_backend() if d.pg else None))
    finally:
        d.close()


def test_two_gloo_ranks_max_and_sum():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, w, mx, sm, backend in got:
        assert w == 2 and backend == "gloo"
        assert mx == 2.5          # max over ranks of 1.5 + rank
        assert sm == 30.0         # 10 + 20


def test_single_process_is_a_no_op():
    os.environ.pop("WORLD_SIZE", None)
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    assert d.world == 1 and d.pg is None
    d.barrier()
    assert d.max(3.0) == 3.0 and d.sum(4.0) == 4.0
