"""The benchmark's multi-rank path on CPU: two gloo ranks, max time over ranks, units summed."""

import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms, units = bench.aggregate(10.0 + rank * 5.0, 1000.0, world)
    bench.barrier(world)
    q.put((rank, ms, units))
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 15.0, 2000.0), (1, 15.0, 2000.0)]


def test_single_rank_aggregate_is_identity():
    import bench

    assert bench.aggregate(3.5, 7.0, 1) == (3.5, 7.0)


def test_work_accounting_for_the_mixed_step():
    import bench
    from continuous_batching_paged_pkv_gb300 import workloads as W

    w = W.mixed(0)
    # chunk rows 1024..1535 see 1025..1536 keys: 4 * D * Hq * sum
    assert bench.chunk_flops(w) == 4 * 128 * 32 * sum(range(1025, 1537))
    assert bench.kv_bytes(w) == sum(s.ctx for s in w.segments) * 8 * 128 * 4 + 516 * 32 * 128 * 4
