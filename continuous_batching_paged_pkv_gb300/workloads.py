"""Seeded synthetic inputs for one paged-KV attention step.

This module only draws random numbers and lays out shapes. It holds none of the
method's arithmetic: no slot mapping, no packing, no attention. The CUDA path's
tests and benchmark and the CPU oracle both consume what it produces, each with
its own arithmetic.

The workloads mirror the serving situations described in the pages:

* Lucebox, "Continuous batching: Qwen3.8-27B at 301 tok/s across five clients,
  up to 1.97x llama.cpp" -- §Paged KV and paged attention (block tables drawn
  from a shared free pool), §Chunked prefill is a slot phase (a 3,000-token
  prompt advanced 512 tokens per step next to decode rows), §Packing unequal
  prompt chunks together (prompt chunks first, decode rows last on one axis).
* mlxcel manual, "Continuous batching" -- §Chunked prefill (2048-token chunks
  with no decoder, 512 while a decode batch runs).

There is no dataset on the pages for this path; every tensor here is N(0, 1)
drawn in float32 and rounded to bfloat16, with sizes chosen per workload.
"""

from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

# Bit pattern of a quiet bfloat16 NaN. Pool rows that no token ever wrote hold
# it, so a kernel that reads past a sequence's history poisons its output.
BF16_NAN_SENTINEL = 0x7FC1


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return uint16 bits.

    Inputs are finite draws, so the carry out of the mantissa never reaches
    the sign bit.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def _rngs(seed: int, n: int, *key: int) -> list[np.random.Generator]:
    ss = np.random.SeedSequence(entropy=seed, spawn_key=tuple(key))
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(n)]


@dataclass
class Segment:
    """One stretch of the packed token axis: ``q_len`` new rows of slot ``slot``.

    ``ctx`` is the slot's context length after this step's rows are appended.
    """

    slot: int
    q_len: int
    ctx: int


@dataclass
class StepInputs:
    """Everything one synthetic step needs, before any lowering.

    ``blocks[slot]`` lists the physical block IDs owned by the slot in logical
    order (a reservation may own more blocks than its context uses).
    ``hist_k[slot]`` / ``hist_v[slot]`` hold the slot's whole key/value history
    ``[ctx, Hkv, D]`` as bfloat16 bits; the last ``q_len`` rows are the ones this
    step appends. ``q`` holds the packed query rows ``[T, Hq, D]``.
    """

    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_slots: int
    max_blocks_per_slot: int
    segments: list[Segment]
    blocks: dict[int, np.ndarray]
    hist_k: dict[int, np.ndarray]
    hist_v: dict[int, np.ndarray]
    q: np.ndarray
    seed: int = 0
    free_order: np.ndarray | None = None  # remaining free stack, top last
    notes: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def total_q(self) -> int:
        return sum(s.q_len for s in self.segments)

    def block_table_array(self) -> np.ndarray:
        """Block tables as an int32 ``[max_slots, max_blocks_per_slot]`` array, -1 unused."""
        bt = np.full((self.max_slots, self.max_blocks_per_slot), -1, dtype=np.int32)
        for slot, ids in self.blocks.items():
            bt[slot, : len(ids)] = ids
        return bt

    def new_k(self) -> np.ndarray:
        """Packed ``[T, Hkv, D]`` keys appended by this step, in segment order."""
        return _concat([self.hist_k[s.slot][s.ctx - s.q_len: s.ctx] for s in self.segments],
                       (0, self.num_kv_heads, self.head_dim))

    def new_v(self) -> np.ndarray:
        return _concat([self.hist_v[s.slot][s.ctx - s.q_len: s.ctx] for s in self.segments],
                       (0, self.num_kv_heads, self.head_dim))

    def kv_bytes(self) -> int:
        """Key+value bytes the step's attention must read once (bf16)."""
        return sum(s.ctx for s in self.segments) * self.num_kv_heads * self.head_dim * 2 * 2


def _concat(parts, empty_shape):
    if not parts:
        return np.zeros(empty_shape, dtype=np.uint16)
    return np.ascontiguousarray(np.concatenate(parts, axis=0))


def _draw_histories(seed, segments, hkv, d, threads):
    """Per-slot K/V histories from per-slot substreams, drawn in parallel."""
    def one(seg):
        rk, rv = _rngs(seed, 2, 1, seg.slot)
        return seg.slot, _normal_bf16(rk, (seg.ctx, hkv, d)), _normal_bf16(rv, (seg.ctx, hkv, d))

    with ThreadPoolExecutor(max_workers=threads or 8) as ex:
        out = list(ex.map(one, segments))
    return {s: k for s, k, _ in out}, {s: v for s, _, v in out}


def _draw_q(seed, total, hq, d):
    (rq,) = _rngs(seed, 1, 2)
    return _normal_bf16(rq, (total, hq, d))


def _finish(name, seed, hq, hkv, d, bs, num_blocks, max_slots, mbps, segments, blocks,
            free_order, threads, notes=None):
    hist_k, hist_v = _draw_histories(seed, segments, hkv, d, threads)
    q = _draw_q(seed, sum(s.q_len for s in segments), hq, d)
    return StepInputs(name=name, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                      num_blocks=num_blocks, max_slots=max_slots, max_blocks_per_slot=mbps,
                      segments=segments, blocks=blocks, hist_k=hist_k, hist_v=hist_v, q=q,
                      seed=seed, free_order=free_order, notes=notes or {})


def _take(free: list[int], n: int) -> np.ndarray:
    """Pop ``n`` block IDs off the top (end) of a free stack."""
    if n > len(free):
        raise RuntimeError(f"synthetic pool exhausted: need {n}, have {len(free)}")
    out = free[len(free) - n:][::-1]
    del free[len(free) - n:]
    return np.asarray(out, dtype=np.int32)


def tiny(seed: int = 0, threads=None) -> StepInputs:
    """Tiny correctness step: 4 q heads / 2 kv heads, head_dim 64, block 16, 32 blocks.

    Slot 0 (A) decodes one row at context 37, slot 1 (B) runs a 16-row causal
    prefill chunk at offset 64, slot 2 (C) decodes one row at context 5. Packed
    prompt first, decode rows after: [B x16][A][C].
    """
    (rt,) = _rngs(seed, 1, 0)
    free = [int(b) for b in rt.permutation(32)]
    segs = [Segment(1, 16, 80), Segment(0, 1, 37), Segment(2, 1, 5)]
    blocks = {0: _take(free, 3), 1: _take(free, 5), 2: _take(free, 1)}
    return _finish("tiny", seed, 4, 2, 64, 16, 32, 4, 8, segs, blocks,
                   np.asarray(free, dtype=np.int32), threads)


def decode5(seed: int = 0, threads=None, pool_blocks: int = 65536) -> StepInputs:
    """Decode-only step, five clients: 40 q / 8 kv heads, head_dim 128, 65,536 blocks.

    Five slots each decode one row; contexts are uniform in [1024, 8192] and
    block tables come off a shuffled free list. ``pool_blocks`` shrinks the
    pool (same contexts, other physical blocks) for profiling captures.
    """
    rt, rl = _rngs(seed, 2, 0)
    free = [int(b) for b in rt.permutation(pool_blocks)]
    ctx = rl.integers(1024, 8193, size=5)
    segs = [Segment(i, 1, int(c)) for i, c in enumerate(ctx)]
    blocks = {s.slot: _take(free, -(-s.ctx // 16)) for s in segs}
    return _finish("decode5", seed, 40, 8, 128, 16, pool_blocks, 8, 512, segs, blocks,
                   np.asarray(free, dtype=np.int32), threads)


def mixed(seed: int = 0, threads=None, pool_blocks: int = 65536) -> StepInputs:
    """Mixed step: 32 q / 8 kv heads, head_dim 128; one 512-row chunk + 4 decode rows.

    Slot 0 runs the chunk [1024, 1536) of a 3000-token prompt; its admission
    reserved ceil(3001 / 16) = 188 blocks. Slots 1-4 decode one row each at
    contexts uniform in [200, 4000]. Packed [chunk x512][d1][d2][d3][d4].
    """
    rt, rl = _rngs(seed, 2, 0)
    free = [int(b) for b in rt.permutation(pool_blocks)]
    ctx = rl.integers(200, 4001, size=4)
    segs = [Segment(0, 512, 1536)] + [Segment(1 + i, 1, int(c)) for i, c in enumerate(ctx)]
    blocks = {0: _take(free, 188)}
    for s in segs[1:]:
        blocks[s.slot] = _take(free, -(-s.ctx // 16))
    return _finish("mixed", seed, 32, 8, 128, 16, pool_blocks, 8, 256, segs, blocks,
                   np.asarray(free, dtype=np.int32), threads,
                   notes={"prompt_len": 3000, "chunk": (1024, 1536)})


def decode256(seed: int = 0, threads=None, pool_blocks: int = 131072) -> StepInputs:
    """Large decode batch: 256 slots, 64 q / 8 kv heads, head_dim 128, 131,072 blocks.

    Contexts are lognormal with median 2048 (sigma 1), clipped to [16, 32768].
    The free list is fragmented first: four rounds each hand out 64 tables of
    1-512 blocks and then free a random half of them in random order; the 256
    tables are then drawn from what the free stack holds.
    """
    rt, rl, rf = _rngs(seed, 3, 0)
    free = [int(b) for b in rt.permutation(pool_blocks)]
    for _ in range(4):
        held = [_take(free, int(n)) for n in rf.integers(1, 513, size=64)]
        for i in rf.permutation(64)[:32]:
            free.extend(int(b) for b in held[i][::-1])
    z = rl.standard_normal(256)
    ctx = np.clip(np.round(2048.0 * np.exp(z)), 16, 32768).astype(np.int64)
    segs = [Segment(i, 1, int(c)) for i, c in enumerate(ctx)]
    blocks = {s.slot: _take(free, -(-s.ctx // 16)) for s in segs}
    return _finish("decode256", seed, 64, 8, 128, 16, pool_blocks, 256, 2048, segs, blocks,
                   np.asarray(free, dtype=np.int32), threads)


def chunk2048(seed: int = 0, threads=None, pool_blocks: int = 65536) -> StepInputs:
    """A prompt chunk of the size taken while nothing decodes: 32 q / 8 kv heads, head_dim 128.

    Slot 0 runs the final chunk [6144, 8192) of an 8,192-token prompt (2,048
    rows, each seeing 6,145 to 8,192 keys); its admission reserved
    ceil(8193 / 16) = 513 blocks, off a shuffled free list of the pool.
    """
    (rt,) = _rngs(seed, 1, 0)
    free = [int(b) for b in rt.permutation(pool_blocks)]
    segs = [Segment(0, 2048, 8192)]
    blocks = {0: _take(free, 513)}
    return _finish("chunk2048", seed, 32, 8, 128, 16, pool_blocks, 1, 520, segs, blocks,
                   np.asarray(free, dtype=np.int32), threads, notes={"prompt_len": 8192, "chunk": (6144, 8192)})


def verify(n: int, seed: int = 0, threads=None, pool_blocks: int = 131072) -> StepInputs:
    """Speculative verification step: 64 slots each check ``n`` draft rows (causal), 32 q / 8 kv heads.

    Contexts after the step are uniform in [1024, 8192]; the n rows of a slot
    sit at its last n positions. Block tables come off a shuffled free list.
    """
    rt, rl = _rngs(seed, 2, 10, n)
    free = [int(b) for b in rt.permutation(pool_blocks)]
    ctx = rl.integers(1024, 8193, size=64)
    segs = [Segment(i, n, int(c)) for i, c in enumerate(ctx)]
    blocks = {s.slot: _take(free, -(-s.ctx // 16)) for s in segs}
    return _finish(f"verify{n}", seed, 32, 8, 128, 16, pool_blocks, 64, 512, segs, blocks,
                   np.asarray(free, dtype=np.int32), threads)


def random_step(seed: int, shapes: list[tuple[int, int]], *, num_q_heads=4, num_kv_heads=2,
                head_dim=64, block_size=16, num_blocks=None, max_slots=None,
                slots: list[int] | None = None, threads=None) -> StepInputs:
    """A small step with given ``(q_len, ctx)`` segments, in the given packed order.

    Slots default to 0..S-1; block tables come off a shuffled free list.
    """
    rt, rs = _rngs(seed, 2, 3)
    nblk = [-(-c // block_size) for _, c in shapes]
    num_blocks = num_blocks or max(1, 2 * sum(nblk))
    max_slots = max_slots or max(len(shapes), 1)
    if slots is None:
        slots = list(range(len(shapes)))
    free = [int(b) for b in rt.permutation(num_blocks)]
    segs = [Segment(sl, ql, c) for sl, (ql, c) in zip(slots, shapes)]
    blocks = {s.slot: _take(free, n) for s, n in zip(segs, nblk)}
    mbps = max(nblk + [1])
    return _finish(f"random{seed}", seed, num_q_heads, num_kv_heads, head_dim, block_size,
                   num_blocks, max_slots, mbps, segs, blocks,
                   np.asarray(free, dtype=np.int32), threads)


WORKLOADS = {"tiny": tiny, "decode5": decode5, "mixed": mixed, "decode256": decode256, "chunk2048": chunk2048,
             "verify4": lambda seed=0, **kw: verify(4, seed, **kw), "verify8": lambda seed=0, **kw: verify(8, seed, **kw),
             "verify16": lambda seed=0, **kw: verify(16, seed, **kw)}


def make_step(name: str, seed: int = 0, threads=None, pool_blocks: int | None = None) -> StepInputs:
    if pool_blocks:
        return WORKLOADS[name](seed, threads=threads, pool_blocks=pool_blocks)
    return WORKLOADS[name](seed, threads=threads)


# ---------------------------------------------------------------------------
# Continuous-batching churn trace (200 steps).
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Request:
    rid: int
    arrival_step: int
    prompt_len: int
    output_len: int
    priority: int = 0  # higher is more urgent
    prefix_id: int = -1  # requests with the same prefix_id share their first prefix_len prompt tokens
    prefix_len: int = 0


@dataclass(frozen=True)
class ChurnSpec:
    num_steps: int = 200
    arrival_rate: float = 2.0
    prompt_min: int = 128
    prompt_max: int = 8192
    output_mean: float = 256.0
    output_max: int = 4096
    num_q_heads: int = 32
    num_kv_heads: int = 8
    head_dim: int = 128
    block_size: int = 16
    num_blocks: int = 131072
    max_slots: int = 64
    high_priority: float = 0.0  # fraction of requests with priority 1 (the rest 0)
    prefix_groups: int = 0      # distinct shared prompt prefixes (0: none)
    prefix_share: float = 0.0   # fraction of requests whose prompt starts with one of them
    prefix_min: int = 64        # shared prefix lengths ~ U[min, max], each below its request's prompt
    prefix_max: int = 512


def churn_trace(seed: int = 0, spec: ChurnSpec = ChurnSpec()) -> list[Request]:
    """Arrivals Poisson(rate) per step; prompt ~ U[min, max]; output ~ Geometric(1/mean), clipped.

    Priorities and shared prefixes come from streams of their own, so the trace
    without them is unchanged. A shared prefix (one of ``prefix_groups``, each
    with a length drawn once) is given to a ``prefix_share`` fraction of the
    requests whose prompt is longer than it."""
    (r,) = _rngs(seed, 1, 4)
    (rp,) = _rngs(seed, 1, 7)
    (rx,) = _rngs(seed, 1, 9)
    plens = [int(rx.integers(spec.prefix_min, spec.prefix_max + 1)) for _ in range(spec.prefix_groups)]
    reqs = []
    for step in range(spec.num_steps):
        for _ in range(int(r.poisson(spec.arrival_rate))):
            p = int(r.integers(spec.prompt_min, spec.prompt_max + 1))
            o = int(min(r.geometric(1.0 / spec.output_mean), spec.output_max))
            prio = int(rp.random() < spec.high_priority) if spec.high_priority > 0 else 0
            pid, plen = -1, 0
            if spec.prefix_groups > 0 and rx.random() < spec.prefix_share:
                g = int(rx.integers(spec.prefix_groups))
                if plens[g] < p:
                    pid, plen = g, plens[g]
            reqs.append(Request(len(reqs), step, p, o, prio, pid, plen))
    return reqs


def churn_free_order(seed: int, num_blocks: int) -> np.ndarray:
    """Initial free stack for the churn pool: a seeded shuffle (top of stack last)."""
    (r,) = _rngs(seed, 1, 5)
    return r.permutation(num_blocks).astype(np.int32)


class TokenSource:
    """Deterministic per-request, per-position K/V/q rows for the churn trace.

    Rows are drawn in pages of 256 positions from a stream keyed by
    (seed, request, page), so a row's value does not depend on how a scheduler
    chunks the prompt. The first ``prefix_len`` positions of a request with a
    shared prefix come from a stream keyed by (seed, prefix, page) instead, so
    every request sharing that prefix has the same rows there.
    """

    PAGE = 256

    def __init__(self, seed: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 cache_pages: int = 512, requests=()):
        self.seed, self.hq, self.hkv, self.d = seed, num_q_heads, num_kv_heads, head_dim
        self._cache: dict = {}
        self._cap = cache_pages
        self._prefix = {r.rid: (r.prefix_id, r.prefix_len) for r in requests if r.prefix_id >= 0}

    def _page(self, rid: int, page: int, shared: bool = False):
        key = ("p" if shared else "r", rid, page)
        hit = self._cache.get(key)
        if hit is not None:
            return hit
        rk, rv, rq = _rngs(self.seed, 3, 8 if shared else 6, rid, page)
        val = (_normal_bf16(rk, (self.PAGE, self.hkv, self.d)),
               _normal_bf16(rv, (self.PAGE, self.hkv, self.d)),
               _normal_bf16(rq, (self.PAGE, self.hq, self.d)))
        if len(self._cache) >= self._cap:
            self._cache.pop(next(iter(self._cache)))
        self._cache[key] = val
        return val

    def rows(self, rid: int, begin: int, end: int):
        """(k, v, q) bf16 bits for positions [begin, end) of request ``rid``."""
        ks, vs, qs = [], [], []
        pos = begin
        pid, plen = self._prefix.get(rid, (-1, 0))
        while pos < end:
            page, off = divmod(pos, self.PAGE)
            take = min(end - pos, self.PAGE - off)
            if pos < plen:
                take = min(take, plen - pos)
                k, v, q = self._page(pid, page, shared=True)
            else:
                k, v, q = self._page(rid, page)
            ks.append(k[off:off + take])
            vs.append(v[off:off + take])
            qs.append(q[off:off + take])
            pos += take
        shape_kv = (0, self.hkv, self.d)
        return (_concat(ks, shape_kv), _concat(vs, shape_kv), _concat(qs, (0, self.hq, self.d)))
