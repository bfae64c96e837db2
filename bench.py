#!/usr/bin/env python
"""Benchmark of the paged-KV attention step (cache write + attention) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload churn|decode5|mixed|decode256|chunk2048|verify4|verify8|verify16|tiny]

Prints one JSON line. The default workload is the continuous-batching churn
trace (arrivals, chunked prompts beside decode rows, retirements; 32 q / 8 kv
heads, head_dim 128, block 16, 131,072-block pool): the decode + prefill mix
the metric is quoted on. Its K timed steps are spread evenly over the trace's
steady state, steps 50 to 199 (a 512-row prompt chunk beside a decode batch
that grows from 6 to over 20 rows), whatever W is; every step of the trace
runs in order, the W steps before step 50 as timed-style warm-up. Metric: KV bytes the attention must read (each
sequence's K and V once per kv head, plus Q in and O out) per second of device
time, and packed rows per second.

The same line carries, under ``configs``, every single-step workload (decode
x5, mixed, decode x256, a 2048-row chunk, verify steps of 4/8/16 rows), each
with its value, roofline, end-to-end figure and oracle CPU baseline, and the
256-row decode step over 8-bit and 4-bit pools.

Timing: before each step a 256 MiB buffer is overwritten (larger than the
129 MB L2) so no step finds its K/V in L2, and a second 256 MiB buffer is then
read so that L2 holds clean lines (otherwise the flush's dirty lines would be
written back inside the timed step). A ~0.2 ms GPU busy-wait follows, during
which the host queues the step's launches, so the events bracket GPU work and
not the host's enqueue time; Python's cyclic garbage collector is off while
steps are timed (a collection inside the enqueue would outlast the busy-wait)
and runs between trace steps instead. All of it is outside the CUDA events
that bracket the step. A second pass times the chunk kernel alone and the decode
and merge kernels alone on the same step (same stream, same flush): the
per-kernel rooflines. Under torchrun (N > 1) every rank runs an independent
replica (the step has no exchange between GPUs); the job's time is the
maximum over ranks.
"""

from __future__ import annotations

import argparse
import contextlib
import gc
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-attn KV GB/s & % of HBM peak; step rows/s (decode + prefill mix)"
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Write a buffer larger than L2, then read another one (clean lines)."""

    def __init__(self, device):
        import torch

        self.dirty = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.clean = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self):
        self.dirty.zero_()
        self.sink.copy_(self.clean.sum())


FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

WORKLOAD_TEXT = {
    "decode5": "decode step, 5 slots x 1 row, 40 q / 8 kv heads, head_dim 128, block 16, "
               "contexts U[1024, 8192], 65,536-block pool",
    "mixed": "mixed step, one 512-row prompt chunk at offset 1024 of a 3000-token prompt + 4 decode rows "
             "(contexts U[200, 4000]), 32 q / 8 kv heads, head_dim 128, block 16, 65,536-block pool",
    "decode256": "decode step, 256 slots x 1 row, 64 q / 8 kv heads, head_dim 128, block 16, "
                 "lognormal contexts (median 2048, clip [16, 32768]), fragmented 131,072-block pool",
    "chunk2048": "prompt chunk, the final 2048 rows [6144, 8192) of an 8192-token prompt, nothing decoding, "
                 "32 q / 8 kv heads, head_dim 128, block 16, 65,536-block pool",
    "verify4": "verify step, 64 slots x 4 causal draft rows, contexts U[1024, 8192], 32 q / 8 kv heads, "
               "head_dim 128, block 16, 131,072-block pool",
    "verify8": "verify step, 64 slots x 8 causal draft rows, contexts U[1024, 8192], 32 q / 8 kv heads, "
               "head_dim 128, block 16, 131,072-block pool",
    "verify16": "verify step, 64 slots x 16 causal draft rows, contexts U[1024, 8192], 32 q / 8 kv heads, "
                "head_dim 128, block 16, 131,072-block pool",
    "tiny": "tiny mixed step, 4 q / 2 kv heads, head_dim 64, block 16, 32 blocks",
    "churn": "continuous-batching trace: Poisson(2) arrivals per step, prompts U[128, 8192], outputs "
             "geometric (mean 256, max 4096), 64 slots, chunks of 512 (2048 while nothing decodes), "
             "32 q / 8 kv heads, head_dim 128, block 16, 131,072-block pool; each step planned by the "
             "library's scheduler, pool and lowering",
}
# Single-step workloads carried in the churn line's ``configs``: (workload, pool format).
EXTRA_CONFIGS = (("decode5", "bf16"), ("mixed", "bf16"), ("decode256", "bf16"), ("chunk2048", "bf16"),
                 ("verify4", "bf16"), ("verify8", "bf16"), ("verify16", "bf16"),
                 ("decode256", "q8"), ("decode256", "q4"))
# Start of the churn trace's steady state: from here a decode batch runs beside
# every 512-row prompt chunk; the timed steps are spread over the rest of the trace.
CHURN_OFFSET = 50
L2_NOTE = ("flushed before every step: 256 MiB written, then 256 MiB read so L2 holds clean lines; "
           "both outside the timed events")


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=150)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOAD_TEXT), default="churn")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle CPU-baseline budget")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=300)
    p.add_argument("--no-configs", action="store_true", help="churn line without the single-step configs")
    p.add_argument("--config-steps", type=int, default=100, help="timed steps of each single-step config")
    p.add_argument("--config-cpu-seconds", type=float, default=2.0)
    p.add_argument("--kv", choices=["bf16", "q8", "q4"], default="bf16",
                   help="pool format: bf16, or the 8-bit / 4-bit block-scaled pool (no end-to-end leg)")
    p.add_argument("--pool-blocks", type=int, default=None,
                   help="smaller synthetic pool (same contexts) for profiling captures")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# Work accounting (from the workload's shapes only).
# ---------------------------------------------------------------------------

def kv_bytes(w, kv: str = "bf16", segments=None) -> int:
    """Algorithmic bytes of the attention: K and V of every visible key once per kv head, Q in, O out.

    A key's row costs 2 * head_dim bytes in a bf16 pool, head_dim (8-bit) or
    head_dim / 2 (4-bit) bytes of codes plus head_dim / 32 bf16 scales in the
    block-scaled pools. ``segments`` restricts the count to those segments."""
    segs = w.segments if segments is None else segments
    codes = {"bf16": 0, "q8": w.head_dim, "q4": w.head_dim // 2}[kv]
    row = w.head_dim * 2 if kv == "bf16" else codes + w.head_dim // 16
    kvb = sum(s.ctx for s in segs) * w.num_kv_heads * row * 2
    return kvb + sum(s.q_len for s in segs) * w.num_q_heads * w.head_dim * 2 * 2


def decode_path(w, s) -> bool:
    """Segments of up to 16 / G rows run on the split-KV decode path, longer ones on the chunk kernel."""
    return s.q_len <= max(1, 16 // (w.num_q_heads // w.num_kv_heads))


def chunk_flops(w) -> int:
    """Causal-only flops of the chunk-path rows: 4 * D * Hq * sum over rows of visible keys."""
    tot = 0
    for s in w.segments:
        if s.q_len > 0 and not decode_path(w, s):
            first = s.ctx - s.q_len + 1
            tot += s.q_len * first + s.q_len * (s.q_len - 1) // 2
    return 4 * w.head_dim * w.num_q_heads * tot


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def profiled_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is unchanged since."""
    src = os.path.join(ROOT, "continuous_batching_paged_pkv_gb300", "csrc", kernel_file)
    summary = os.path.join(ROOT, "profiles", f"{os.path.splitext(kernel_file)[0]}_{workload}.md")
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        for line in open(summary):
            if line.startswith("TRAFFIC "):
                fields = dict(kv.split("=", 1) for kv in line.split()[1:])
                if fields.get("source_sha") == sha:
                    return int(fields["bytes_per_launch"])
    except OSError:
        pass
    return None


# ---------------------------------------------------------------------------
# Clocks during the timed region.
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    @classmethod
    def for_device(cls, dev):
        import torch

        props = torch.cuda.get_device_properties(dev)
        uuid = str(getattr(props, "uuid", "")) or None
        return cls(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else uuid)

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        # nvidia-smi's start-up (its driver queries) must not overlap the timed
        # region: wait for its first sample, for at most 10 s
        t0 = time.perf_counter()
        while self.proc is not None and self.proc.poll() is None and time.perf_counter() - t0 < 10.0:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.05)
        time.sleep(0.4)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        self.proc.wait(timeout=10)
        rows = [r.split(", ") for r in open(self.path).read().strip().splitlines() if r.strip()]
        os.unlink(self.path)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for nm, val in zip(names, r[5:9]):
                if val.strip() == "Active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# Multi-rank plumbing (replicas: one independent step per GPU).
# ---------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def aggregate(local_ms: float, local_units: float, world: int):
    """Max time over ranks, units summed over ranks (every rank does the same work)."""
    if world == 1:
        return local_ms, local_units
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def mean(xs):
    return sum(xs) / len(xs)


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on the host's cores.
# ---------------------------------------------------------------------------

def cpu_baseline(w, seconds: float, threads=None):
    """The oracle on whole steps of ``w`` (paged walk, fp64) for about ``seconds``."""
    import oracle

    oracle.build()
    cores = threads or oracle.default_threads()
    st = oracle.prepare_step(w)
    done_bytes, runs = 0, 0
    t0 = time.perf_counter()
    while True:
        oracle.step_attention(w, st, threads=cores)
        done_bytes += kv_bytes(w)
        runs += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": done_bytes / el / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{runs} run(s) of the oracle over the whole step in {el:.1f} s (fp64, {cores} threads)"}


def churn_oracle_rows(samples, toks, hkv, hq, d, scale, seconds, threads=None):
    """The oracle's dense attention on sampled churn rows (a segment's last row
    over its whole history), about ``seconds`` of oracle time on ``threads``
    host threads, one row per thread at a time. Up to two rows per thread,
    spread evenly over the samples, have their histories generated once
    (outside the clock); the timed loop cycles over them."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    oracle.build()
    cores = threads or oracle.default_threads()
    keep = max(1, min(len(samples), 2 * cores))
    picked = [samples[(i * len(samples)) // keep] for i in range(keep)]
    rows = [(toks.rows(rid, 0, L), qrow, L) for rid, L, qrow in picked]
    done_b, runs, el = 0, 0, 0.0
    with ThreadPoolExecutor(max_workers=cores) as ex:
        while el < seconds:
            for b0 in range(0, len(rows), cores):
                batch = rows[b0:b0 + cores]
                t0 = time.perf_counter()
                list(ex.map(lambda it: oracle.attention_dense(it[1], it[0][0], it[0][1], scale), batch))
                el += time.perf_counter() - t0
                done_b += sum(L * hkv * d * 4 + hq * d * 4 for _, _, L in batch)
                runs += len(batch)
                if el >= seconds:
                    break
    return {"value": done_b / el / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{runs} runs over {len(rows)} sampled rows of the timed trace steps (the last row of a "
                      f"segment, over its whole history), fp64, {cores} threads one row each, {el:.1f} s of "
                      f"oracle time"}


# ---------------------------------------------------------------------------
# Reference arm: the oracle on the host.
# ---------------------------------------------------------------------------

def run_reference(args, rank, world):
    """The oracle timed on the host as the reference arm (rank 0 only)."""
    if rank != 0:
        return None
    from continuous_batching_paged_pkv_gb300 import workloads as W
    import oracle

    oracle.build()
    if args.workload == "churn":
        return run_reference_churn(args)
    w = W.make_step(args.workload, args.seed)
    st = oracle.prepare_step(w)
    cores = oracle.default_threads()
    segs, start = [], 0
    for s in w.segments:
        segs.append((start, s))
        start += s.q_len

    # Each step is one segment of the workload (rotating), so K steps stay bounded.
    def one(i):
        r0, s = segs[i % len(segs)]
        oracle.step_attention(w, st, rows=list(range(r0, r0 + s.q_len)), threads=cores)
        return s.ctx * w.num_kv_heads * w.head_dim * 4 + s.q_len * w.num_q_heads * w.head_dim * 4

    for i in range(args.warmup):
        one(i)
    total_b, t0 = 0, time.perf_counter()
    for i in range(args.steps):
        total_b += one(i)
    el = time.perf_counter() - t0
    val = total_b / el / 1e9
    return {"metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el * 1e3 / max(args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT[args.workload]}",
                       "sample": "one segment of the step per timed step, rotating"},
            "impl": "reference",
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} steps of one segment each, fp64, {cores} threads"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def churn_window(args, num_steps):
    """The trace steps to time: K = --steps of them, spread evenly over the
    steady-state range [CHURN_OFFSET, num_steps) (every step of it when K covers
    the range; the window moves earlier when K is larger still). Every step runs
    in trace order; the W steps before the first timed one are timed-style
    warm-up."""
    timed = max(1, min(args.steps, num_steps))
    first = min(CHURN_OFFSET, num_steps - timed)
    span = num_steps - first
    return [first + (i * span) // timed for i in range(timed)]


def describe_window(steps, num_steps, warmup):
    first = steps[0]
    every = "every step of" if len(steps) == num_steps - first else f"{len(steps)} steps spread evenly over"
    return (f"steps 0..{first - 1} replayed untimed (the last {min(warmup, first)} as timed-style warm-up); "
            f"{every} {first}..{num_steps - 1} timed ({', '.join(map(str, steps[:4]))}, ..., {steps[-1]})"
            + ("" if every.startswith("every") else ", the steps between them replayed untimed"))


def run_reference_churn(args):
    """The churn trace as the oracle replays it (its own admission rules, no
    library code); rows of the timed window sampled as in the churn arm."""
    import numpy as np

    from oracle import churn
    from continuous_batching_paged_pkv_gb300 import workloads as W

    spec = W.ChurnSpec()
    reqs = W.churn_trace(args.seed, spec)
    ref = churn.ChurnReplay(reqs, max_slots=spec.max_slots, num_blocks=spec.num_blocks, block_size=spec.block_size)
    toks = W.TokenSource(args.seed, spec.num_q_heads, spec.num_kv_heads, spec.head_dim)
    window = churn_window(args, spec.num_steps)
    timed_set = set(window)
    samples = []
    for step in range(window[-1] + 1):
        rows = ref.plan()
        if step in timed_set:
            for r in rows:
                samples.append((r.rid, r.begin + r.n, toks.rows(r.rid, r.begin + r.n - 1, r.begin + r.n)[2]))
        ref.commit(rows)
    cb = churn_oracle_rows(samples, toks, spec.num_kv_heads, spec.num_q_heads, spec.head_dim,
                           1.0 / np.sqrt(spec.head_dim), args.cpu_seconds)
    return {"metric": METRIC, "value": cb["value"], "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"churn: {WORKLOAD_TEXT['churn']}",
                       "trace_steps": describe_window(window, spec.num_steps, args.warmup), "sample": cb["sample"]},
            "impl": "reference", "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------
# Our arm: single steps.
# ---------------------------------------------------------------------------

# GPU cycles of busy-wait between the L2 flush and the first event of a timed
# call (~0.2 ms at 2 GHz): the host queues every launch of the call while it
# runs, so the events bracket the call's GPU work and not the host's enqueue
# time (which the end-to-end leg measures).
QUEUE_SPIN_CYCLES = 400_000
QUEUE_NOTE = "every timed call queued behind a ~0.2 ms GPU busy-wait after the flush, before its first event"


@contextlib.contextmanager
def gc_paused():
    """Python's cyclic garbage collector off, after one full collection. A
    collection that lands inside a timed call stalls the host for about a
    millisecond while it enqueues the step, many times a short step's length
    (reference counting still frees everything that is not in a cycle)."""
    was = gc.isenabled()
    gc.collect()
    gc.disable()
    try:
        yield
    finally:
        if was:
            gc.enable()


def timed_calls(flush, stream, fns, n):
    """Run ``fns`` ``n`` times, each time after an L2 flush and a short GPU
    busy-wait, with events between the calls: per call, a list of ``n``
    durations in ms."""
    import torch

    out = [[] for _ in fns]
    chunk = 500
    done = 0
    while done < n:
        m = min(chunk, n - done)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)] for _ in range(m)]
        for row in ev:
            flush()
            torch.cuda._sleep(QUEUE_SPIN_CYCLES)
            row[0].record(stream)
            for f, e in zip(fns, row[1:]):
                f()
                e.record(stream)
        torch.cuda.synchronize()
        for row in ev:
            for i in range(len(fns)):
                out[i].append(row[i].elapsed_time(row[i + 1]))
        done += m
    return out


def measure_step(name, w, dev, **kw):
    """Device and end-to-end timings of one synthetic step (see the module docstring)."""
    with gc_paused():
        return _measure_step(name, w, dev, **kw)


def _measure_step(name, w, dev, *, kv, steps, warmup, e2e_steps, flush, world=1, clocks=False):
    import torch

    from continuous_batching_paged_pkv_gb300 import binding as B
    from continuous_batching_paged_pkv_gb300 import runtime as R

    ds = R.prepare(w, dev, kv=kv)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush()
        R.run_step(ds)
    torch.cuda.synchronize()
    if B.pkv_check_device_status(ds.status) != 0:
        raise RuntimeError(f"{name}: device status reported an error during warm-up")

    sampler = ClockSampler.for_device(dev) if clocks else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    # Timed region: one event pair around each whole step (cache write + attention).
    (step_ms,) = timed_calls(flush, stream, [lambda: (R.run_cache_write(ds), R.run_attention(ds))], steps)
    torch.cuda.synchronize()
    barrier(world)
    clk = sampler.stop() if sampler else None
    # Breakdown pass (same stream, same flush): each call's own duration.
    nb = max(steps // 4, 20)
    write_ms, attn_ms = timed_calls(flush, stream, [lambda: R.run_cache_write(ds), lambda: R.run_attention(ds)], nb)
    # Per-kernel passes: the same attention call with only the chunk items (the
    # chunk kernel alone), and with only the decode and merge items.
    chunk_ms = decode_ms = []
    if kv == "bf16":
        cw, dw = R.split_work(ds.work, ds.info)
        if cw is not None:
            (chunk_ms,) = timed_calls(flush, stream, [lambda: R.run_chunk_only(ds, cw)], nb)
        if dw is not None:
            (decode_ms,) = timed_calls(flush, stream, [lambda: R.run_decode_only(ds, dw)], nb)
    if B.pkv_check_device_status(ds.status) != 0:
        raise RuntimeError(f"{name}: device status reported an error during the timed steps")
    e2e = run_e2e(w, ds, dev, flush, e2e_steps) if kv == "bf16" else None
    info = ds.info
    launches = (int(w.total_q > 0) + int(info.num_decode_items > 0) + int(info.num_prefill_items > 0)
                + int(info.num_combine_items > 0))
    del ds
    torch.cuda.empty_cache()
    return {"step_ms": step_ms, "write_ms": write_ms, "attn_ms": attn_ms, "chunk_ms": chunk_ms,
            "decode_ms": decode_ms, "e2e": e2e, "clocks": clk, "launches": launches}


def kernel_rooflines(w, m, kv, hbm, tflops, peak_src, workload):
    """Per-kernel figures: the chunk kernel against the bf16 peak, the decode
    and merge kernels against HBM. Returns (dict by kernel, the dominant one)."""
    out = {}
    if m["chunk_ms"]:
        cm = mean(m["chunk_ms"])
        fl = chunk_flops(w)
        ach = fl / (cm / 1e3) / 1e12
        src = "pkv_prefill_pair.cu" if w.head_dim == 128 else "pkv_prefill.cu"
        out["chunk"] = {"bound": "tensor", "kernel": "prefill_pair_kernel" if w.head_dim == 128 else "prefill_kernel",
                        "achieved": ach, "peak": tflops, "unit": "TFLOP/s", "frac": ach / tflops,
                        "traffic": profiled_traffic(src, workload), "algorithmic_flop_per_launch": fl,
                        "mean_launch_ms": cm,
                        "peak_source": f"{peak_src} bf16 burst (the chunk kernel is timed alone)"}
    if m["decode_ms"]:
        dm = mean(m["decode_ms"])
        db = kv_bytes(w, kv, [s for s in w.segments if s.q_len > 0 and decode_path(w, s)])
        ach = db / (dm / 1e3) / 1e9
        quant = kv in ("q8", "q4")
        dec = "decode_quant_kernel" if quant else "decode_kernel"
        src, wl = ("pkv_kvquant.cu", f"{workload}_{kv}") if quant else ("pkv_decode.cu", workload)
        out["decode"] = {"bound": "hbm", "kernel": f"{dec} + span merge (merge_small/merge_wide)",
                         "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                         "traffic": profiled_traffic(src, wl) if not m["chunk_ms"] else None,
                         "algorithmic_bytes_per_launch": db, "mean_launch_ms": dm,
                         "peak_source": f"{peak_src} HBM copy bandwidth"}
    if not out:
        return out, None
    dominant = max(out, key=lambda k: out[k]["mean_launch_ms"])
    return out, dominant


def single_line(name, w, m, *, kv, world, steps, cpu=None):
    """The metric and its rooflines for one synthetic step workload."""
    hbm, tflops, peak_src = peaks()
    kvb = kv_bytes(w, kv)
    total_ms, total_bytes = aggregate(sum(m["step_ms"]), kvb * steps, world)
    value = total_bytes / (total_ms / 1e3) / 1e9
    attn_mean = mean(m["attn_ms"])
    achieved = kvb / (attn_mean / 1e3) / 1e9
    res = {
        "value": value, "unit": "GB/s", "ms_per_step": total_ms / steps,
        "pct_hbm_peak": 100.0 * value / world / hbm,
        "rows_per_s": world * w.total_q / (total_ms / steps / 1e3),
        "step_breakdown_ms": {"cache_write": statistics.median(m["write_ms"]),
                              "attention": statistics.median(m["attn_ms"]),
                              "step": statistics.median(m["step_ms"])},
        "attention_call": {"kv_gbs": achieved, "pct_hbm_peak": 100.0 * achieved / hbm, "mean_ms": attn_mean},
    }
    kernels, dominant = kernel_rooflines(w, m, kv, hbm, tflops, peak_src, name)
    if kernels:
        res["kernels"] = kernels
    decode_only = all(decode_path(w, s) for s in w.segments if s.q_len > 0)
    if dominant == "chunk":
        res["roofline"] = kernels["chunk"]
    elif (dominant == "decode" and "chunk" not in kernels) or (dominant is None and decode_only):
        # decode-only steps: the attention call (decode + merge) is the kernel pair that bounds the step
        dec = "decode_quant_kernel" if kv in ("q8", "q4") else "decode_kernel"
        src = "pkv_kvquant.cu" if kv in ("q8", "q4") else "pkv_decode.cu"
        wl = name if kv == "bf16" else f"{name}_{kv}"
        res["roofline"] = {"bound": "hbm", "kernel": f"attention call: {dec} + span merge (merge_small/merge_wide)",
                           "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                           "traffic": profiled_traffic(src, wl), "algorithmic_bytes_per_launch": kvb,
                           "mean_launch_ms": attn_mean, "peak_source": f"{peak_src} HBM copy bandwidth"}
    elif dominant == "decode":
        res["roofline"] = kernels["decode"]
    else:
        res["roofline"] = {"bound": "hbm", "kernel": "attention call", "achieved": achieved, "peak": hbm,
                           "unit": "GB/s", "frac": achieved / hbm, "traffic": None,
                           "algorithmic_bytes_per_launch": kvb, "mean_launch_ms": attn_mean,
                           "peak_source": f"{peak_src} HBM copy bandwidth"}
    if m["e2e"]:
        e = m["e2e"]
        e_ms, e_units = aggregate(e["ms_total"], kvb * e["steps"], world)
        res["e2e"] = {"value": e_units / (e_ms / 1e3) / 1e9, "unit": "GB/s",
                      "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                      "steps": e["steps"], "ms_per_step": e_ms / e["steps"],
                      "timed": "wall clock per step: one pkv_step call (work list planned on the host, "
                               + ("the staged inputs read by the kernels in place from pinned host memory"
                                  if e["in_place"] else "H2D copy of the staged inputs")
                               + ", cache write, attention, "
                               + ("the output written by the kernels straight to pinned host memory"
                                  if e["out_direct"] else "D2H copy of the output")
                               + ") and the stream synchronised"}
    if cpu:
        res["cpu_baseline"] = cpu
    return res


def run_ours(args, rank, world, local_rank):
    import torch

    from continuous_batching_paged_pkv_gb300 import build as libbuild
    from continuous_batching_paged_pkv_gb300 import workloads as W

    libbuild.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = W.make_step(args.workload, args.seed, pool_blocks=args.pool_blocks)
    flush = L2Flush(dev)
    m = measure_step(args.workload, w, dev, kv=args.kv, steps=args.steps, warmup=args.warmup,
                     e2e_steps=args.e2e_steps, flush=flush, world=world, clocks=True)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)
        one = cpu_baseline(w, args.cpu_seconds / 2, threads=1)  # the same oracle on one core
        cpu["one_core"] = {"value": one["value"], "unit": one["unit"], "sample": one["sample"]}
    line = single_line(args.workload, w, m, kv=args.kv, world=world, steps=args.steps, cpu=cpu)
    res = {"metric": METRIC, "value": line.pop("value"), "unit": line.pop("unit"), "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": line.pop("ms_per_step"),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT[args.workload]}",
                      "rows_per_step": w.total_q, "kv_bytes_per_step": kv_bytes(w, args.kv), "kv_format": args.kv,
                      "l2": L2_NOTE, "queue": QUEUE_NOTE, "parallelism": f"replicas x{world} (no exchange between GPUs)",
                      "seed": args.seed, "pool_blocks": w.num_blocks}}
    res.update(line)
    res["gpu_launches"] = m["launches"] * args.steps
    res["clocks"] = m["clocks"]
    res["impl"] = "ours"
    return res


def run_configs(args, rank, world, dev, flush):
    """Every single-step workload, each with its own figures (for the churn line's ``configs``)."""
    import torch

    from continuous_batching_paged_pkv_gb300 import workloads as W

    out = {}
    steps = max(args.config_steps, 20)
    for name, kv in EXTRA_CONFIGS:
        key = name if kv == "bf16" else f"{name}_{kv}"
        w = W.make_step(name, args.seed)
        try:
            m = measure_step(name, w, dev, kv=kv, steps=steps, warmup=max(args.warmup, 3),
                             e2e_steps=min(args.e2e_steps, 100), flush=flush, world=world)
        except (RuntimeError, MemoryError) as e:
            if world > 1:
                raise  # the ranks' barriers must stay paired
            # one configuration's failure (say, no room for its pool) is reported in the
            # line instead of taking the churn figures down with it
            out[key] = {"workload": WORKLOAD_TEXT[name], "error": f"{type(e).__name__}: {e}"[:300]}
            del w
            torch.cuda.empty_cache()
            continue
        cpu = None
        if rank == 0 and world == 1 and not args.no_cpu_baseline and kv == "bf16":
            cpu = cpu_baseline(w, args.config_cpu_seconds)
        line = single_line(name, w, m, kv=kv, world=world, steps=steps, cpu=cpu)
        line["workload"] = WORKLOAD_TEXT[name]
        line["steps"] = steps
        if kv != "bf16":
            # KV GB/s counts the pool's own bytes (codes and group scales)
            line["kv_format"] = kv
            line["kv_bytes_per_step"] = kv_bytes(w, kv)
            line["e2e"] = None
            line["note"] = ("quantised pool: the host-staged one-call path (e2e) serves bf16 pools only; the "
                            "oracle baseline is on the bf16 line of the same workload")
        out[key] = line
        del w
        torch.cuda.empty_cache()
    return out


def run_e2e(w, ds, dev, flush, e2e_steps):
    """The step through the one-call host path: the inputs sit in a page-locked
    staging buffer; the timed region is ``pkv_step`` (work list planned on the
    host, the H2D copy, cache write, attention, the D2H copy of the output),
    called through ``binding.StepCall`` (arguments bound once, as a serving loop
    reusing its buffers would), and the stream synchronisation. With
    PKV_STEP_IN_PLACE the kernels write the output straight to the pinned host
    buffer instead of the copy out, and small steps without prompt chunks read
    their inputs in place instead of the copy in."""
    import torch

    from continuous_batching_paged_pkv_gb300 import binding as B
    from continuous_batching_paged_pkv_gb300 import runtime as R

    if e2e_steps <= 0:
        return None
    low = ds.lowered
    lay = B.pkv_stage_layout_init(w.total_q, len(w.segments), w.max_slots, w.max_blocks_per_slot, w.num_q_heads,
                                  w.num_kv_heads, w.head_dim)
    stage = R.HostStage(lay.work + 4 * int(ds.info.work_words), dev)
    stage.fill(lay, q=w.q, k_new=w.new_k(), v_new=w.new_v(), slot_mapping=low.slot_mapping,
               cu_seqlens_q=low.cu_seqlens_q, seq_slot=low.seq_slot, context_lens=low.context_lens,
               block_tables=ds.pool.block_tables())
    out_host = torch.empty(ds.out.shape, dtype=torch.bfloat16, pin_memory=True)
    h2d = lay.work + 4 * int(ds.info.work_words)
    d2h = out_host.numel() * 2
    stream = torch.cuda.current_stream()
    step = B.StepCall(lay, stage.host, stage.device, ds.k_pool, ds.v_pool, ds.out, ds.workspace, out_host=out_host,
                      scale=w.scale, device_status=ds.status, stream=stream, in_place=True)
    times = []
    for i in range(e2e_steps + 5):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        info = step()
        stream.synchronize()
        if i >= 5:
            times.append((time.perf_counter() - t0) * 1e3)
    if B.pkv_check_device_status(ds.status) != 0:
        raise RuntimeError("device status reported an error in the end-to-end steps")
    out_direct = True
    in_place = info.num_prefill_items == 0 and h2d <= B.PKV_STEP_IN_PLACE_MAX_BYTES
    return {"ms_total": sum(times), "steps": len(times), "h2d": h2d, "d2h": d2h, "in_place": in_place,
            "out_direct": out_direct}


# ---------------------------------------------------------------------------
# Our arm: the churn trace.
# ---------------------------------------------------------------------------

def run_churn(args, rank, world, local_rank):
    """The churn trace replayed through the library: every step runs (the pool
    state is the trace's), host planning outside the events, cache write +
    attention inside (L2 flushed first); steps before the window are untimed."""
    import numpy as np
    import torch

    from continuous_batching_paged_pkv_gb300 import binding as B
    from continuous_batching_paged_pkv_gb300 import build as libbuild
    from continuous_batching_paged_pkv_gb300 import runtime as R
    from continuous_batching_paged_pkv_gb300 import scheduler as S
    from continuous_batching_paged_pkv_gb300 import workloads as W

    libbuild.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    spec = W.ChurnSpec()
    if args.pool_blocks:
        spec = W.ChurnSpec(num_blocks=args.pool_blocks)
    reqs = W.churn_trace(args.seed, spec)
    bs, hq, hkv, d = spec.block_size, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    mbps = -(-(spec.prompt_max + spec.output_max + 1) // bs) + 1
    pool = B.Pool(spec.num_blocks, bs, spec.max_slots, mbps, free_order=W.churn_free_order(args.seed, spec.num_blocks))
    sch = S.ChurnScheduler(reqs, pool)
    toks = W.TokenSource(args.seed, hq, hkv, d)
    k_pool, v_pool = R.empty_pool(spec.num_blocks, hkv, bs, d, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    scale = 1.0 / np.sqrt(d)
    window = churn_window(args, spec.num_steps)
    timed_set, first = set(window), window[0]
    sample_cpu = not args.no_cpu_baseline and rank == 0 and world == 1
    cpu_rows = []  # (request, length, last q row) of timed segments, for the oracle baseline

    step_ms, e2e_ms, step_bytes, step_rows = [], [], [], []
    chunk_ms, chunk_fl, dec_ms, dec_bytes, write_ms, attn_ms = [], [], [], [], [], []
    prefill_steps = launches = h2d_tot = d2h_tot = 0
    clocks = stage = ws = None
    with gc_paused():
        for step in range(window[-1] + 1):
            gc.collect()  # outside every timed region; the collector is off inside them
            rows = sch.plan()
            if not rows:
                sch.commit(rows)
                continue
            low = pool.lower([(r.slot, r.n) for r in rows])
            parts = [toks.rows(r.rid, r.begin, r.begin + r.n) for r in rows]
            host = {"k": np.concatenate([p[0] for p in parts]), "v": np.concatenate([p[1] for p in parts]),
                    "q": np.concatenate([p[2] for p in parts])}
            T = len(host["q"])
            lay = B.pkv_stage_layout_init(T, len(rows), spec.max_slots, mbps, hq, hkv, d)
            # sizing only (outside the timed region): the step plans its own work list again inside
            _, info0 = B.pkv_plan_work(low.cu_seqlens_q, low.seq_slot, low.context_lens, max_slots=spec.max_slots,
                                       max_blocks_per_slot=mbps, block_size=bs, num_q_heads=hq, num_kv_heads=hkv,
                                       head_dim=d)
            need = lay.work + 4 * int(info0.work_words)
            if stage is None or stage.nbytes < need:
                stage = R.HostStage(max(need, 32 << 20), dev)
            if ws is None or ws.numel() < int(info0.workspace_bytes):
                ws = torch.empty(max(int(info0.workspace_bytes), 64 << 20), dtype=torch.uint8, device=dev)
            stage.fill(lay, q=host["q"], k_new=host["k"], v_new=host["v"], slot_mapping=low.slot_mapping,
                       cu_seqlens_q=low.cu_seqlens_q, seq_slot=low.seq_slot, context_lens=low.context_lens,
                       block_tables=pool.block_tables())
            out = torch.empty((T, hq, d), dtype=torch.bfloat16, device=dev)
            out_host = torch.empty(out.shape, dtype=torch.bfloat16, pin_memory=True)
            ctx = [int(low.context_lens[r.slot]) for r in rows]
            nbytes = sum(ctx) * hkv * d * 4 + T * hq * d * 4
            is_timed = step in timed_set
            is_warm = is_timed or first - args.warmup <= step < first
            if is_timed and clocks is None:
                clocks = ClockSampler.for_device(dev)
                clocks.start()

            # end to end: one pkv_step call (work list, H2D, both calls, output straight to host), synchronised
            flush()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            info = B.pkv_step(lay, stage.host, stage.device, k_pool, v_pool, out, ws, out_host=out_host, scale=scale,
                              device_status=status, stream=stream, in_place=True)
            stream.synchronize()
            e2e = (time.perf_counter() - t0) * 1e3

            # device time of the step alone (inputs resident in the device stage), same calls again
            v = stage.device_views(lay, info)

            def write():
                B.pkv_cache_write(v["k_new"], v["v_new"], v["slot_mapping"], k_pool, v_pool, device_status=status)

            def attend(work=v["work"], inf=info, space=ws):
                B.pkv_attention(v["q"], v["cu_seqlens_q"], v["seq_slot"], v["context_lens"], v["block_tables"],
                                k_pool, v_pool, work, inf, out, space, scale=scale, device_status=status)

            if is_warm:
                (st_ms,) = timed_calls(flush, stream, [lambda: (write(), attend())], 1)
            else:
                write()
                attend()
            if is_timed:
                # breakdown: the two calls apart, then the chunk kernel alone and the decode + merge kernels alone
                w_ms, a_ms = timed_calls(flush, stream, [write, attend], 1)
                cw, dw = R.split_work(v["work"], info)
                c_ms = timed_calls(flush, stream, [lambda: attend(cw[0], cw[1], None)], 1)[0] if cw else []
                d_ms = timed_calls(flush, stream, [lambda: attend(dw[0], dw[1], ws)], 1)[0] if dw else []
            torch.cuda.synchronize()
            if B.pkv_check_device_status(status) != 0:
                raise RuntimeError(f"device status reported an error at churn step {step}")
            if is_timed:
                step_ms.extend(st_ms)
                write_ms.extend(w_ms)
                attn_ms.extend(a_ms)
                e2e_ms.append(e2e)
                step_bytes.append(nbytes)
                step_rows.append(T)
                dec_rows = [(r, c) for r, c in zip(rows, ctx) if r.n <= max(1, 16 // (hq // hkv))]
                chk_rows = [(r, c) for r, c in zip(rows, ctx) if r.n > max(1, 16 // (hq // hkv))]
                if c_ms:
                    chunk_ms.extend(c_ms)
                    chunk_fl.append(4 * d * hq * sum(r.n * (c - r.n + 1) + r.n * (r.n - 1) // 2 for r, c in chk_rows))
                if d_ms:
                    dec_ms.extend(d_ms)
                    dec_bytes.append(sum(c for _, c in dec_rows) * hkv * d * 4 + sum(r.n for r, _ in dec_rows) * hq * d * 4)
                prefill_steps += int(any(r.prefill for r in rows))
                launches += 1 + int(info.num_decode_items > 0) + int(info.num_prefill_items > 0) + \
                    int(info.num_combine_items > 0)
                h2d_tot += lay.work + 4 * int(info.work_words)
                d2h_tot += out_host.numel() * 2
            if sample_cpu and is_timed:
                cpu_rows.extend((r.rid, r.begin + r.n, p[2][-1:]) for r, p in zip(rows, parts))
            sch.commit(rows)
    clk = clocks.stop() if clocks is not None else {}

    n = len(step_ms)
    tot_ms, tot_bytes = aggregate(sum(step_ms), sum(step_bytes), world)
    hbm, tflops, peak_src = peaks()
    value = tot_bytes / (tot_ms / 1e3) / 1e9
    e_ms, _ = aggregate(sum(e2e_ms), sum(step_bytes), world)
    kernels = {}
    if chunk_ms:
        ach = sum(chunk_fl) / (sum(chunk_ms) / 1e3) / 1e12
        kernels["chunk"] = {"bound": "tensor", "kernel": "prefill_pair_kernel", "achieved": ach, "peak": tflops,
                            "unit": "TFLOP/s", "frac": ach / tflops,
                            "traffic": profiled_traffic("pkv_prefill_pair.cu", "churn"),
                            "algorithmic_flop_per_launch": sum(chunk_fl) / len(chunk_fl),
                            "mean_launch_ms": mean(chunk_ms), "launches": len(chunk_ms),
                            "total_ms": sum(chunk_ms),
                            "peak_source": f"{peak_src} bf16 burst (the chunk kernel is timed alone, per step)"}
    if dec_ms:
        ach = sum(dec_bytes) / (sum(dec_ms) / 1e3) / 1e9
        kernels["decode"] = {"bound": "hbm", "kernel": "decode_kernel + span merge (merge_small/merge_wide)",
                             "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                             "traffic": profiled_traffic("pkv_decode.cu", "churn"),
                             "algorithmic_bytes_per_launch": sum(dec_bytes) / len(dec_bytes),
                             "mean_launch_ms": mean(dec_ms), "launches": len(dec_ms), "total_ms": sum(dec_ms),
                             "peak_source": f"{peak_src} HBM copy bandwidth (decode and merge kernels timed "
                                            f"alone, per step)"}
    dominant = max(kernels, key=lambda k: kernels[k]["total_ms"]) if kernels else None
    roofline = dict(kernels[dominant]) if dominant else {
        "bound": "hbm", "kernel": "whole step", "achieved": value / world, "peak": hbm, "unit": "GB/s",
        "frac": value / world / hbm, "traffic": None}
    res = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": n, "warmup": args.warmup,
        "ms_per_step": tot_ms / n, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"churn: {WORKLOAD_TEXT['churn']}",
                   "trace_steps": describe_window(window, spec.num_steps, args.warmup),
                   "timed_steps": window,
                   "steps_with_prompt_chunks": prefill_steps, "rows_per_step_mean": sum(step_rows) / n,
                   "kv_bytes_per_step_mean": sum(step_bytes) / n,
                   "step_ms_p50": statistics.median(step_ms), "step_ms_p90": sorted(step_ms)[int(0.9 * (n - 1))],
                   "step_ms_max": max(step_ms), "l2": L2_NOTE, "queue": QUEUE_NOTE,
                   "parallelism": f"replicas x{world} (no exchange between GPUs)", "seed": args.seed,
                   "pool_blocks": spec.num_blocks},
        "pct_hbm_peak": 100.0 * value / world / hbm,
        "rows_per_s": world * sum(step_rows) / (tot_ms / 1e3),
        "step_breakdown_ms": {"cache_write": mean(write_ms), "attention": mean(attn_ms), "step": mean(step_ms),
                              "chunk_kernel_alone": mean(chunk_ms) if chunk_ms else None,
                              "decode_and_merge_alone": mean(dec_ms) if dec_ms else None},
        "roofline": roofline, "kernels": kernels, "roofline_kernel": dominant,
        "gpu_launches": launches, "clocks": clk,
        "e2e": {"value": tot_bytes / (e_ms / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d_tot // n,
                "d2h_bytes_per_step": d2h_tot // n, "steps": n, "ms_per_step": e_ms / n,
                "timed": "wall clock per step: one pkv_step call with PKV_STEP_IN_PLACE (work list planned on "
                         "the host, H2D copy of the staged inputs, cache write, attention, the output written by "
                         "the kernels straight to pinned host memory) and the stream synchronised (K/V/q "
                         "generation, scheduling and staging outside)"},
        "impl": "ours",
    }
    if cpu_rows:
        res["cpu_baseline"] = churn_oracle_rows(cpu_rows, toks, hkv, hq, d, scale, args.cpu_seconds)
    del k_pool, v_pool, stage, ws
    torch.cuda.empty_cache()
    if not args.no_configs and args.kv == "bf16":
        res["configs"] = run_configs(args, rank, world, dev, flush)
    return res


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if args.impl == "reference":
            backend = "gloo"
        dist.init_process_group(backend=backend)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    elif args.workload == "churn":
        res = run_churn(args, rank, world, local_rank)
    else:
        res = run_ours(args, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
