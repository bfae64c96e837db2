#!/usr/bin/env python
"""Benchmark of one paged-KV attention step (cache write + attention) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode5|mixed|decode256|tiny]

Prints one JSON line. The default workload is one decode step for five
clients (40 q / 8 kv heads, head_dim 128, block 16, contexts U[1024, 8192],
65,536-block pool). Metric: KV bytes the attention must read (each sequence's
K and V once per kv head, plus Q in and O out) per second of device time.

Timing: W untimed warm-up steps, then K timed steps. Before each step a
256 MiB buffer is overwritten (larger than the 129 MB L2) so no step finds its
K/V in L2, and a second 256 MiB buffer is then read so that L2 holds clean
lines (otherwise the flush's dirty lines would be written back to HBM inside
the timed step). Both are outside the CUDA events that bracket the step. The
timed region brackets whole steps only, so the step's kernels may overlap
their launches; a second pass brackets each library call with its own events
on the launching stream to give the attention call's own duration (the
roofline figure) and the per-call breakdown. Under torchrun (N > 1) every rank
runs an independent replica (the step has no exchange between GPUs); the
job's time is the maximum over ranks.
"""

from __future__ import annotations

import argparse
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
    "tiny": "tiny mixed step, 4 q / 2 kv heads, head_dim 64, block 16, 32 blocks",
    "churn": "continuous-batching trace: Poisson(2) arrivals per step, prompts U[128, 8192], outputs "
             "geometric (mean 256, max 4096), 64 slots, chunks of 512 (2048 while nothing decodes), "
             "32 q / 8 kv heads, head_dim 128, block 16, 131,072-block pool; each step planned by the "
             "library's scheduler, pool and lowering",
}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=4000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOAD_TEXT), default="decode5")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle CPU-baseline budget")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=300)
    p.add_argument("--kv", choices=["bf16", "q8", "q4"], default="bf16",
                   help="pool format: bf16, or the 8-bit / 4-bit block-scaled pool (no end-to-end leg)")
    p.add_argument("--pool-blocks", type=int, default=None,
                   help="smaller synthetic pool (same contexts) for profiling captures")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# Work accounting (from the workload's shapes only).
# ---------------------------------------------------------------------------

def kv_bytes(w, kv: str = "bf16") -> int:
    """Algorithmic bytes of the attention: K and V of every visible key once per kv head, Q in, O out.

    A key's row costs 2 * head_dim bytes in a bf16 pool, head_dim (8-bit) or
    head_dim / 2 (4-bit) bytes of codes plus head_dim / 32 bf16 scales in the
    block-scaled pools."""
    codes = {"bf16": 0, "q8": w.head_dim, "q4": w.head_dim // 2}[kv]
    row = w.head_dim * 2 if kv == "bf16" else codes + w.head_dim // 16
    kvb = sum(s.ctx for s in w.segments) * w.num_kv_heads * row * 2
    return kvb + w.total_q * w.num_q_heads * w.head_dim * 2 * 2


def write_bytes(w) -> int:
    return w.total_q * w.num_kv_heads * w.head_dim * 2 * 2 * 2  # K+V read and written


def chunk_flops(w) -> int:
    """Causal-only flops of the prompt-chunk rows: 4 * D * Hq * sum over rows of visible keys."""
    tot = 0
    for s in w.segments:
        if s.q_len > 1:
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


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on the host's cores.
# ---------------------------------------------------------------------------

def cpu_baseline(w, seconds: float, rows_per_run=None, threads=None):
    import oracle

    oracle.build()
    cores = threads or oracle.default_threads()
    st = oracle.prepare_step(w)
    seg_rows = []
    start = 0
    for s in w.segments:
        seg_rows.append((start, s))
        start += s.q_len
    done_bytes, runs = 0, 0
    t0 = time.perf_counter()
    while True:
        if rows_per_run is None:
            oracle.step_attention(w, st, threads=cores)
            done_bytes += kv_bytes(w)
        else:
            r0, s = seg_rows[runs % len(seg_rows)]
            oracle.step_attention(w, st, rows=list(range(r0, r0 + s.q_len)), threads=cores)
            done_bytes += s.ctx * w.num_kv_heads * w.head_dim * 4 + s.q_len * w.num_q_heads * w.head_dim * 4
        runs += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": done_bytes / el / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{runs} run(s) of the oracle over " +
                      ("the whole step" if rows_per_run is None else "one segment at a time, in turn") +
                      f" in {el:.1f} s (fp64, {cores} threads)"}


# ---------------------------------------------------------------------------
# Arms.
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


def run_reference_churn(args):
    """The churn trace as the oracle replays it (its own admission rules, no
    library code); each timed step's rows sampled as in the churn arm."""
    import numpy as np

    from oracle import churn
    from continuous_batching_paged_pkv_gb300 import workloads as W

    spec = W.ChurnSpec()
    reqs = W.churn_trace(args.seed, spec)
    ref = churn.ChurnReplay(reqs, max_slots=spec.max_slots, num_blocks=spec.num_blocks, block_size=spec.block_size)
    toks = W.TokenSource(args.seed, spec.num_q_heads, spec.num_kv_heads, spec.head_dim)
    warm = max(args.warmup, 3)
    samples = []
    for step in range(warm + max(1, min(args.steps, spec.num_steps - warm))):
        rows = ref.plan()
        if step >= warm:
            for r in rows:
                samples.append((r.rid, r.begin + r.n, toks.rows(r.rid, r.begin + r.n - 1, r.begin + r.n)[2]))
        ref.commit(rows)
    cb = churn_oracle_rows(samples, toks, spec.num_kv_heads, spec.num_q_heads, spec.head_dim,
                           1.0 / np.sqrt(spec.head_dim), args.cpu_seconds)
    return {"metric": METRIC, "value": cb["value"], "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"churn: {WORKLOAD_TEXT['churn']}", "sample": cb["sample"]},
            "impl": "reference", "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    from continuous_batching_paged_pkv_gb300 import binding as B
    from continuous_batching_paged_pkv_gb300 import build as libbuild
    from continuous_batching_paged_pkv_gb300 import runtime as R
    from continuous_batching_paged_pkv_gb300 import workloads as W

    libbuild.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = W.make_step(args.workload, args.seed, pool_blocks=args.pool_blocks)
    ds = R.prepare(w, dev, kv=args.kv)
    stream = torch.cuda.current_stream()
    kvb = kv_bytes(w, args.kv)
    flush = L2Flush(dev)
    launches_per_step = (int(w.total_q > 0) + int(ds.info.num_decode_items > 0) + int(ds.info.num_prefill_items > 0)
                         + int(ds.info.num_combine_items > 0))

    for _ in range(args.warmup):
        flush()
        R.run_step(ds)
    torch.cuda.synchronize()
    if B.pkv_check_device_status(ds.status) != 0:
        raise RuntimeError("device status reported an error during warm-up")

    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "")) or None
    clocks = ClockSampler(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else uuid)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    # Timed region: one event pair around each whole step (cache write +
    # attention), so the step's kernels may overlap their launches.
    step_ms = []
    chunk = 500
    done = 0
    while done < args.steps:
        n = min(chunk, args.steps - done)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for e0, e2 in ev:
            flush()
            e0.record(stream)
            R.run_cache_write(ds)
            R.run_attention(ds)
            e2.record(stream)
        torch.cuda.synchronize()
        step_ms.extend(e0.elapsed_time(e2) for e0, e2 in ev)
        done += n
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    # Breakdown pass (same stream, same flush): events between the two calls
    # give each call's own duration; the attention call is the roofline kernel.
    write_ms, attn_ms = [], []
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(max(args.steps // 4, 20))]
    for e0, e1, e2 in ev:
        flush()
        e0.record(stream)
        R.run_cache_write(ds)
        e1.record(stream)
        R.run_attention(ds)
        e2.record(stream)
    torch.cuda.synchronize()
    for e0, e1, e2 in ev:
        write_ms.append(e0.elapsed_time(e1))
        attn_ms.append(e1.elapsed_time(e2))
    # Chunk-kernel pass: the same call with only the prompt-chunk items of the
    # work list launches the tensor-core chunk kernel alone (same inputs and
    # output rows), so its own duration is measured on the launching stream.
    chunk_ms = []
    if ds.info.num_prefill_items and args.kv == "bf16":
        wi = R.chunk_only(ds)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(max(args.steps // 4, 20))]
        for e0, e1 in ev:
            flush()
            e0.record(stream)
            R.run_chunk_only(ds, wi)
            e1.record(stream)
        torch.cuda.synchronize()
        chunk_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    if B.pkv_check_device_status(ds.status) != 0:
        raise RuntimeError("device status reported an error during the timed steps")

    total_ms, total_bytes = aggregate(sum(step_ms), kvb * args.steps, world)
    hbm, tflops, peak_src = peaks()
    value = total_bytes / (total_ms / 1e3) / 1e9
    attn_mean = sum(attn_ms) / len(attn_ms)
    achieved = kvb / (attn_mean / 1e3) / 1e9
    res = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT[args.workload]}",
                   "rows_per_step": w.total_q, "kv_bytes_per_step": kvb, "kv_format": args.kv,
                   "l2": "flushed before every step: 256 MiB written, then 256 MiB read so L2 holds clean lines; "
                         "both outside the timed events",
                   "parallelism": f"replicas x{world} (no exchange between GPUs)", "seed": args.seed,
                   "pool_blocks": w.num_blocks},
        "pct_hbm_peak": 100.0 * value / world / hbm,
        "rows_per_s": world * w.total_q / (total_ms / args.steps / 1e3),
        "step_breakdown_ms": {"cache_write": statistics.median(write_ms), "attention": statistics.median(attn_ms),
                              "step": statistics.median(step_ms)},
    }
    chunk_kernel = "prefill_pair_kernel" if w.head_dim == 128 else "prefill_kernel"
    dec_kernel = "decode_quant_kernel" if args.kv in ("q8", "q4") else "decode_kernel"
    if ds.info.num_prefill_items and args.kv == "bf16":
        # the chunk kernel dominates the library's time on steps that carry a prompt chunk
        bound, unit, kernel = "tensor", "TFLOP/s", chunk_kernel
    elif ds.info.num_prefill_items:
        bound, unit, kernel = "hbm", "GB/s", "attention call: widen_quant + chunk + decode_quant + span merge kernels"
    elif ds.info.num_combine_items:
        bound, unit, kernel = "hbm", "GB/s", f"attention call: {dec_kernel} + span merge (merge_small/merge_wide)"
    else:
        bound, unit, kernel = "hbm", "GB/s", dec_kernel
    if bound == "tensor":
        chunk_mean = sum(chunk_ms) / len(chunk_ms)
        ach = chunk_flops(w) / (chunk_mean / 1e3) / 1e12
        src = "pkv_prefill_pair.cu" if w.head_dim == 128 else "pkv_prefill.cu"
        res["roofline"] = {"bound": "tensor", "kernel": kernel, "achieved": ach, "peak": tflops,
                           "unit": "TFLOP/s", "frac": ach / tflops, "traffic": profiled_traffic(src, args.workload),
                           "algorithmic_flop_per_launch": chunk_flops(w), "mean_launch_ms": chunk_mean,
                           "peak_source": f"{peak_src} bf16 burst (the chunk kernel is timed alone)"}
        res["attention_call"] = {"kv_gbs": achieved, "pct_hbm_peak": 100.0 * achieved / hbm, "mean_ms": attn_mean,
                                 "kernels": "chunk + decode + span merge"}
    else:
        src = "pkv_kvquant.cu" if args.kv in ("q8", "q4") else "pkv_decode.cu"
        wl = args.workload if args.kv == "bf16" else f"{args.workload}_{args.kv}"
        traffic = profiled_traffic(src, wl) if dec_kernel in kernel else None
        res["roofline"] = {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                           "frac": achieved / hbm, "traffic": traffic,
                           "algorithmic_bytes_per_launch": kvb, "mean_launch_ms": attn_mean,
                           "peak_source": f"{peak_src} HBM copy bandwidth"}
    if chunk_ms:
        res["chunk_kernel_ms"] = statistics.median(chunk_ms)
    res["gpu_launches"] = launches_per_step * args.steps
    res["clocks"] = clk

    # ---- end to end through the C ABI, inputs from pinned host memory ----
    e2e = run_e2e(args, w, ds, dev, flush) if args.kv == "bf16" else None
    if e2e:
        e_ms, e_units = aggregate(e2e["ms_total"], kvb * e2e["steps"], world)
        res["e2e"] = {"value": e_units / (e_ms / 1e3) / 1e9, "unit": "GB/s",
                      "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                      "steps": e2e["steps"], "ms_per_step": e_ms / e2e["steps"],
                      "timed": "wall clock per step: one pkv_step call (work list planned on the host, "
                               "one H2D copy of the staged inputs, cache write, attention, one D2H copy of "
                               "the output) and the stream synchronised"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
        one = cpu_baseline(w, args.cpu_seconds / 2, threads=1)  # the same oracle on one core
        res["cpu_baseline"]["one_core"] = {"value": one["value"], "unit": one["unit"], "sample": one["sample"]}
    res["impl"] = "ours"
    return res


def run_e2e(args, w, ds, dev, flush):
    """The step through the one-call host path: the inputs sit in a page-locked
    staging buffer; the timed region is ``pkv_step`` (work list planned on the
    host, one H2D copy, cache write, attention, one D2H copy of the output),
    called through ``binding.StepCall`` (arguments bound once, as a serving loop
    reusing its buffers would), and the stream synchronisation."""
    import torch

    from continuous_batching_paged_pkv_gb300 import binding as B
    from continuous_batching_paged_pkv_gb300 import runtime as R

    if args.e2e_steps <= 0:
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
                      scale=w.scale, device_status=ds.status, stream=stream)
    times = []
    for i in range(args.e2e_steps + 5):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step()
        stream.synchronize()
        if i >= 5:
            times.append((time.perf_counter() - t0) * 1e3)
    if B.pkv_check_device_status(ds.status) != 0:
        raise RuntimeError("device status reported an error in the end-to-end steps")
    return {"ms_total": sum(times), "steps": len(times), "h2d": h2d, "d2h": d2h}


def run_churn(args, rank, world, local_rank):
    """The churn trace replayed through the library: host planning per step
    outside the events, cache write + attention inside (L2 flushed first)."""
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
    warm = max(args.warmup, 3)
    timed = max(1, min(args.steps, spec.num_steps - warm))
    sample_cpu = not args.no_cpu_baseline and rank == 0 and world == 1
    cpu_rows = []  # (request, length, last q row) of timed segments, for the oracle baseline

    step_ms, e2e_ms, step_bytes, step_rows, prefill_steps = [], [], [], [], 0
    launches = h2d_tot = d2h_tot = 0
    clocks = stage = ws = None
    for step in range(warm + timed):
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
        ctx = sum(int(low.context_lens[r.slot]) for r in rows)
        nbytes = ctx * hkv * d * 4 + T * hq * d * 4
        is_timed = step >= warm
        if is_timed and clocks is None:
            props = torch.cuda.get_device_properties(dev)
            uuid = str(getattr(props, "uuid", "")) or None
            clocks = ClockSampler(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else uuid)
            clocks.start()

        # end to end: one pkv_step call (work list, H2D, both calls, D2H), synchronised
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        info = B.pkv_step(lay, stage.host, stage.device, k_pool, v_pool, out, ws, out_host=out_host, scale=scale,
                          device_status=status, stream=stream)
        stream.synchronize()
        e2e = (time.perf_counter() - t0) * 1e3

        # device time of the step alone (inputs resident in the device stage), same calls again
        v = stage.device_views(lay, info)
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        B.pkv_cache_write(v["k_new"], v["v_new"], v["slot_mapping"], k_pool, v_pool, device_status=status)
        B.pkv_attention(v["q"], v["cu_seqlens_q"], v["seq_slot"], v["context_lens"], v["block_tables"], k_pool,
                        v_pool, v["work"], info, out, ws, scale=scale, device_status=status)
        e1.record(stream)
        torch.cuda.synchronize()
        if B.pkv_check_device_status(status) != 0:
            raise RuntimeError(f"device status reported an error at churn step {step}")
        if is_timed:
            step_ms.append(e0.elapsed_time(e1))
            e2e_ms.append(e2e)
            step_bytes.append(nbytes)
            step_rows.append(T)
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
    hbm, _, peak_src = peaks()
    value = tot_bytes / (tot_ms / 1e3) / 1e9
    e_ms, _ = aggregate(sum(e2e_ms), sum(step_bytes), world)
    res = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": n, "warmup": warm,
        "ms_per_step": tot_ms / n, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"churn: {WORKLOAD_TEXT['churn']}",
                   "trace_steps": f"{warm} untimed, then {n} timed, of {spec.num_steps}",
                   "steps_with_prompt_chunks": prefill_steps, "rows_per_step_mean": sum(step_rows) / n,
                   "step_ms_p50": statistics.median(step_ms), "step_ms_p90": sorted(step_ms)[int(0.9 * (n - 1))],
                   "step_ms_max": max(step_ms),
                   "l2": "flushed before every step (256 MiB written, then 256 MiB read), outside the events",
                   "parallelism": f"replicas x{world} (no exchange between GPUs)", "seed": args.seed,
                   "pool_blocks": spec.num_blocks},
        "pct_hbm_peak": 100.0 * value / world / hbm,
        "rows_per_s": world * sum(step_rows) / (tot_ms / 1e3),
        "roofline": {"bound": "hbm", "kernel": "whole step (cache write + attention call), summed over the trace",
                     "achieved": value / world, "peak": hbm, "unit": "GB/s", "frac": value / world / hbm,
                     "traffic": None, "algorithmic_bytes_per_launch": sum(step_bytes) / n,
                     "mean_launch_ms": sum(step_ms) / n, "peak_source": f"{peak_src} HBM copy bandwidth"},
        "gpu_launches": launches, "clocks": clk,
        "e2e": {"value": tot_bytes / (e_ms / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d_tot // n,
                "d2h_bytes_per_step": d2h_tot // n, "steps": n, "ms_per_step": e_ms / n,
                "timed": "wall clock per step: one pkv_step call (work list planned on the host, one H2D "
                         "copy of the staged inputs, cache write, attention, one D2H copy of the output) and "
                         "the stream synchronised (K/V/q generation, scheduling and staging outside)"},
        "impl": "ours",
    }
    if cpu_rows:
        res["cpu_baseline"] = churn_oracle_rows(cpu_rows, toks, hkv, hq, d, scale, args.cpu_seconds)
    return res


def churn_oracle_rows(samples, toks, hkv, hq, d, scale, seconds):
    """The oracle's dense attention on sampled churn rows (a segment's last row
    over its whole history), spread evenly over the samples, ~`seconds` of work."""
    import oracle

    oracle.build()
    stride = max(1, len(samples) // 400)
    done_b, runs, el = 0, 0, 0.0
    for rid, L, qrow in samples[::stride]:
        k, v, _ = toks.rows(rid, 0, L)  # the history, generated outside the clock
        t0 = time.perf_counter()
        oracle.attention_dense(qrow, k, v, scale)
        el += time.perf_counter() - t0
        done_b += L * hkv * d * 4 + hq * d * 4
        runs += 1
        if el >= seconds:
            break
    return {"value": done_b / el / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{runs} sampled rows of the timed trace steps (the last row of a segment, over its "
                      f"whole history), fp64, one thread, {el:.1f} s of oracle time"}


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
