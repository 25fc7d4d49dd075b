"""The N > 1 path of bench.py on CPU: two gloo ranks (replicas), a barrier
and the max-over-ranks timing feeding the whole-job throughput."""
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


def _rank(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    ctx = bench.DistCtx(backend="gloo")
    ctx.barrier()
    my_ms = 100.0 + 50.0 * rank  # rank 1 is the slow one
    worst = ctx.max(my_ms)
    value = bench.aggregate_throughput(2.0 * 4096 ** 3, 10, ctx.world, worst)
    ctx.barrier()
    ctx.close()
    q.put((rank, worst, value))


def test_two_gloo_ranks_take_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, worst, value in res:
        assert worst == 150.0
        # 2 replicas x 10 steps x 2*4096^3 FLOP over 150 ms
        assert value == pytest.approx(2 * 10 * 2.0 * 4096 ** 3 / 0.150 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ctx = bench.DistCtx()
    assert ctx.world == 1 and ctx.pg is None
    assert ctx.max(3.5) == 3.5
    assert bench.aggregate_throughput(1e12, 1, 1, 1000.0) == pytest.approx(1.0)
