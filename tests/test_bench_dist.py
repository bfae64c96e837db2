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


def test_gc_is_paused_inside_and_restored_after():
    import gc

    import bench

    assert gc.isenabled()
    with bench.gc_paused():
        assert not gc.isenabled()
    assert gc.isenabled()
    gc.disable()
    try:
        with bench.gc_paused():
            assert not gc.isenabled()
        assert not gc.isenabled(), "a collector that was off stays off"
    finally:
        gc.enable()


def test_clock_sampler_waits_for_the_first_sample(tmp_path, monkeypatch):
    """A stand-in for nvidia-smi that needs a second before its first sample: start()
    returns only after that sample, and stop() reads the clocks and event reasons."""
    import time

    import bench

    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\nsleep 1\n"
                    "while true; do echo '0, 2070, 2070, 812.5, 0x4, Not Active, Not Active, Not Active, Active'; "
                    "sleep 0.1; done\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    sampler = bench.ClockSampler(None)
    t0 = time.perf_counter()
    sampler.start()
    assert time.perf_counter() - t0 >= 1.0
    assert os.path.getsize(sampler.path) > 0
    clk = sampler.stop()
    assert clk["sm_mhz"] == 2070.0 and clk["sm_max_mhz"] == 2070.0
    assert clk["reasons"] == ["sw_power_cap"] and clk["samples"] >= 3


def test_a_failed_config_is_reported_not_fatal(monkeypatch):
    """One configuration that cannot run (here every one: the measurement raises) leaves an
    error entry under its key; the line still forms."""
    import types

    import bench
    from continuous_batching_paged_pkv_gb300 import workloads as W

    monkeypatch.setattr(W, "make_step", lambda name, seed=0, **kw: types.SimpleNamespace(name=name))

    def boom(name, w, dev, **kw):
        raise MemoryError(f"no room for the {kw['kv']} pool of {name}")

    monkeypatch.setattr(bench, "measure_step", boom)
    args = types.SimpleNamespace(config_steps=20, warmup=3, e2e_steps=0, no_cpu_baseline=True, seed=0)
    out = bench.run_configs(args, 0, 1, "cpu", flush=None)
    assert set(out) == {n if kv == "bf16" else f"{n}_{kv}" for n, kv in bench.EXTRA_CONFIGS}
    assert out["decode256_q8"]["error"] == "MemoryError: no room for the q8 pool of decode256"
