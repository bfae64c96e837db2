"""Oracle replay of a continuous-batching trace -- TEST INFRASTRUCTURE.

Only tests, the smoke check and the benchmark's CPU-baseline leg use this. It
decides, step by step, which rows each request contributes, keeping only a
count of free blocks and slots (no physical block IDs), and it keeps each
request's key/value history as one contiguous array. The library's scheduler,
allocator and lowering must produce the same rows, and its paged attention the
same outputs.

Rules, each from the pages (the numeric choices marked "reading" are this
oracle's plain reading where the pages leave a value open):

* Admission needs a free slot plus KV capacity for the prompt and decode
  headroom, reserved atomically; the deferred queue is strict FIFO, so a
  request that does not fit blocks the ones behind it.
  (Lucebox, "Continuous batching ...", §Admission and step planning are
  different decisions.) Reading: the reservation is ceil((prompt + 1) / block)
  blocks, i.e. the prompt plus the first decode row.
* Prefill chunk budget: 2048 tokens while no sequence decodes, 512 while a
  decode batch runs. (mlxcel manual, "Continuous batching", §Chunked prefill.)
  The budget is shared FIFO across prefilling requests, several chunks pack
  into one step, prompt chunks first, decode rows after. (Lucebox §Packing
  unequal prompt chunks together.)
* A request stays in the prefill phase until its last chunk; it decodes from
  the next step on. (Lucebox §Chunked prefill is a slot phase.)
* The final prefill chunk yields the first output token; each decode row
  yields one more. A request retires at the end of the step that produced its
  last output token, returning its slot and blocks at once. (Tutorial 15,
  "Continuous Batching and Scheduling", §4 Chunked Prefill and §6 Request
  Lifecycle; Lucebox §One scheduler, model-specific execution.)
* Decode rows take one more block when their position crosses into a block
  the reservation did not cover.

Budget rules (mlxcel manual, "Continuous batching", §Preemptive eviction,
§Paged KV cache and prefix sharing, and the section on decode headroom under a
tight budget), used only when switched on:

* Watermark F: while some request decodes, the queue head is admitted only if
  free blocks - F * (pool blocks) >= its reservation.
* Preemption for priority: if the head does not fit (slot or blocks) and some
  admitted request has a strictly lower priority, one of those is evicted --
  policy "longest-first": the one with the most generated tokens;
  "lowest-priority": the lowest priority, most generated tokens on ties --
  and admission is tried again. Reading: remaining ties go to the latest
  admitted.
* Decode headroom: before the step, the blocks that decode rows open must be
  free; otherwise the eviction ladder runs: cold cached prefixes first (with a
  prefix cache, below), then prefixes adopted by waiting requests (none here:
  a waiting request holds no blocks), then admitted requests are preempted,
  least progress first (reading: fewest generated tokens, then fewest cached
  rows, then latest admitted), until they fit.
* A preempted request frees its slot and blocks, keeps its generated-token
  count, and waits again in arrival order; once admitted it prefills its
  prompt plus the tokens it had generated, the last chunk yielding one more
  token, then decodes.

Prompt-prefix cache (mlxcel manual, §Paged KV cache and prefix sharing:
requests sharing a prompt prefix store its blocks once and adopt them by
reference; an adopter is charged only for the blocks its suffix creates; under
a budget, cold cached prefixes are evicted, least recently used first, before
anyone is preempted), used only with a capacity C > 0. Readings:

* The cached part of a request's shared prefix of length p is its whole
  blocks, c = floor(p / block) * block tokens (nothing when c = 0), so no
  block is ever shared partly filled and nobody appends into a shared block.
* Donation, at the end of a step before that step's retirements: each request
  (admission order) that prefilled its shared prefix itself and whose position
  has reached c, and whose prefix is not cached, donates its first c / block
  blocks to a new entry; with C entries already cached, the least recently
  used is dropped first. An entry is used when created and when adopted.
* Admission: a head whose prefix is cached adopts the entry's blocks and
  starts prefilling at position c; it needs ceil((rows + 1) / block) - c /
  block fresh blocks. When the head lacks blocks (not a slot), cold entries --
  held by the cache alone, other than the head's own -- are evicted least
  recently used first (ties: the earlier created), until it fits, before
  priority preemption is tried.
* A shared block returns to the free list when its last holder (the entry or
  a request) lets go; an adopter whose entry was dropped keeps the blocks.
"""

from __future__ import annotations

from collections import deque
from dataclasses import dataclass

import numpy as np

from . import attention_dense


@dataclass
class _Entry:
    """A cached prompt prefix: ``nb`` shared blocks and the count of their holders."""

    pid: int
    nb: int
    refs: int
    last_used: int
    order: int


@dataclass
class _Live:
    rid: int
    prompt: int
    output: int
    pos: int = 0
    decoding: bool = False
    generated: int = 0
    blocks: int = 0  # blocks of its own (shared prefix blocks are counted once, in their entry)
    own_prompt: int = 0
    arrival: int = 0
    priority: int = 0
    admitted_as: int = 0
    prefix_id: int = -1
    cached_len: int = 0  # the whole-block part of its shared prefix
    entry: _Entry | None = None  # the shared blocks it holds (adopted or donated)

    @property
    def all_blocks(self) -> int:
        return self.blocks + (self.entry.nb if self.entry else 0)


@dataclass(frozen=True)
class Row:
    """One segment of a step: ``n`` rows of request ``rid`` at positions begin..begin+n-1."""

    rid: int
    begin: int
    n: int
    prefill: bool


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


class ChurnReplay:
    def __init__(self, requests, *, max_slots: int, num_blocks: int, block_size: int,
                 chunk_idle: int = 2048, chunk_busy: int = 512, watermark: float = 0.0,
                 preemption: str | None = None, prefix_cache: int = 0):
        self.pending = deque(sorted(requests, key=lambda r: (r.arrival_step, r.rid)))
        # waiting requests: (arrival, rid, rows to prefill, own prompt, output, priority, generated)
        self.queue: list[tuple] = []
        self.live: list[_Live] = []  # admission order
        self.free_slots = max_slots
        self.free_blocks = num_blocks
        self.num_blocks = num_blocks
        self.bs = block_size
        self.chunk_idle, self.chunk_busy = chunk_idle, chunk_busy
        self.watermark, self.preemption = watermark, preemption
        self.step_index = 0
        self.finished: list[int] = []
        self.preempted: list[int] = []
        self.preempt_reasons: list[str] = []  # "priority" or "headroom"
        self._admissions = 0
        self.cache_capacity = prefix_cache
        self.cache: dict[int, _Entry] = {}
        self._entries_made = 0
        # (step, event, prefix id): "donate", "adopt", "drop-capacity", "drop-admission", "drop-headroom"
        self.cache_events: list[tuple] = []

    # ---- blocks held by requests and cached prefixes --------------------------------
    def _unref(self, e: _Entry) -> None:
        e.refs -= 1
        if e.refs == 0:
            self.free_blocks += e.nb

    def _release(self, r: _Live) -> None:
        self.free_blocks += r.blocks
        if r.entry is not None:
            self._unref(r.entry)

    def _drop(self, e: _Entry, why: str) -> None:
        del self.cache[e.pid]
        self.cache_events.append((self.step_index, "drop-" + why, e.pid))
        self._unref(e)

    def _cold(self, spare: int | None = None) -> list[_Entry]:
        """Cached entries held by the cache alone, least recently used first."""
        cold = [e for e in self.cache.values() if e.refs == 1 and e.pid != spare]
        return sorted(cold, key=lambda e: (e.last_used, e.order))

    def _cached_len(self, prefix_id: int, prefix_len: int) -> int:
        return (prefix_len // self.bs) * self.bs if self.cache_capacity > 0 and prefix_id >= 0 else 0

    def _evict(self, r: _Live, reason: str, held=None) -> None:
        """Free r's slot and blocks; it waits again (in `held` until the request that evicted it is in)."""
        self.live.remove(r)
        self.free_slots += 1
        self._release(r)
        entry = (r.arrival, r.rid, r.own_prompt + r.generated, r.own_prompt, r.output, r.priority, r.generated,
                 r.prefix_id, r.cached_len)
        if held is None:
            self.queue.append(entry)
            self.queue.sort()
        else:
            held.append(entry)
        self.preempted.append(r.rid)
        self.preempt_reasons.append(reason)

    def plan(self) -> list[Row]:
        """Advance admission for the current step and return its rows (packed order)."""
        s = self.step_index
        while self.pending and self.pending[0].arrival_step <= s:
            q = self.pending.popleft()
            pid = getattr(q, "prefix_id", -1)
            self.queue.append((q.arrival_step, q.rid, q.prompt_len, q.prompt_len, q.output_len,
                               getattr(q, "priority", 0), 0, pid,
                               self._cached_len(pid, getattr(q, "prefix_len", 0))))
            self.queue.sort()
        held: list[tuple] = []  # evicted for the current head; they wait behind it
        while self.queue:
            arrival, rid, rows_to_fill, own, output, prio, gen, pid, clen = self.queue[0]
            e = self.cache.get(pid) if clen > 0 else None
            need = _ceil_div(rows_to_fill + 1, self.bs) - (e.nb if e else 0)
            floor = self.watermark * self.num_blocks if any(r.decoding for r in self.live) else 0.0
            if self.free_slots == 0 or self.free_blocks - need < floor:
                cold = self._cold(spare=pid if e else None) if self.free_slots > 0 else []
                if cold:  # first rung: a cold cached prefix
                    self._drop(cold[0], "admission")
                    continue
                lower = [r for r in self.live if r.priority < prio] if self.preemption else []
                if not lower:
                    break  # strict FIFO: nobody jumps ahead
                if self.preemption == "lowest-priority":
                    lower.sort(key=lambda r: (r.priority, -r.generated, -r.admitted_as))
                else:  # longest-first
                    lower.sort(key=lambda r: (-r.generated, -r.admitted_as))
                self._evict(lower[0], "priority", held)
                continue
            self.queue.pop(0)
            if held:
                self.queue.extend(held)
                self.queue.sort()
                held.clear()
            self.free_slots -= 1
            self.free_blocks -= need
            r = _Live(rid, rows_to_fill, output, generated=gen, blocks=need, own_prompt=own, arrival=arrival,
                      priority=prio, admitted_as=self._admissions, prefix_id=pid, cached_len=clen)
            if e is not None:  # adopt: start after the cached prefix
                e.refs += 1
                e.last_used = s
                r.entry, r.pos = e, clen
                self.cache_events.append((s, "adopt", pid))
            self.live.append(r)
            self._admissions += 1
        if held:  # the head still did not fit after every eviction it could make
            self.queue.extend(held)
            self.queue.sort()
        # decode headroom
        while True:
            opening = sum(1 for r in self.live if r.decoding and r.pos // self.bs >= r.all_blocks)
            if opening <= self.free_blocks:
                break
            cold = self._cold()
            if cold:
                self._drop(cold[0], "headroom")
                continue
            self._evict(sorted(self.live, key=lambda r: (r.generated, r.pos, -r.admitted_as))[0], "headroom")
        budget = self.chunk_busy if any(r.decoding for r in self.live) else self.chunk_idle
        rows: list[Row] = []
        for r in self.live:
            if budget == 0:
                break
            if not r.decoding and r.pos < r.prompt:
                take = min(r.prompt - r.pos, budget)
                rows.append(Row(r.rid, r.pos, take, True))
                budget -= take
        for r in self.live:
            if r.decoding:
                if r.pos // self.bs >= r.all_blocks:
                    if self.free_blocks == 0:
                        raise RuntimeError("pool exhausted during decode")
                    self.free_blocks -= 1
                    r.blocks += 1
                rows.append(Row(r.rid, r.pos, 1, False))
        return rows

    def commit(self, rows: list[Row]) -> list[int]:
        """Apply the step's effects; returns the request IDs retired at its end."""
        by_rid = {r.rid: r for r in self.live}
        done = []
        for row in rows:
            r = by_rid[row.rid]
            r.pos += row.n
            if row.prefill:
                if r.pos == r.prompt:
                    r.decoding = True
                    r.generated += 1
            else:
                r.generated += 1
            if r.pos >= r.prompt and r.generated >= r.output:
                done.append(r.rid)
        # donations, before this step's retirements
        for r in self.live:
            if (r.cached_len > 0 and r.entry is None and r.pos >= r.cached_len
                    and r.prefix_id not in self.cache):
                if len(self.cache) >= self.cache_capacity:
                    self._drop(min(self.cache.values(), key=lambda e: (e.last_used, e.order)), "capacity")
                e = _Entry(r.prefix_id, r.cached_len // self.bs, 2, self.step_index, self._entries_made)
                self._entries_made += 1
                self.cache[r.prefix_id] = e
                r.blocks -= e.nb
                r.entry = e
                self.cache_events.append((self.step_index, "donate", r.prefix_id))
        for rid in done:
            r = by_rid[rid]
            self.live.remove(r)
            self.free_slots += 1
            self._release(r)
        self.finished.extend(done)
        self.step_index += 1
        return done


class ContiguousHistory:
    """Each request's keys/values as one growing [L, Hkv, D] array (no pool)."""

    def __init__(self):
        self.k: dict[int, list] = {}
        self.v: dict[int, list] = {}
        self.len: dict[int, int] = {}

    def append(self, rid: int, k: np.ndarray, v: np.ndarray) -> None:
        self.k.setdefault(rid, []).append(k)
        self.v.setdefault(rid, []).append(v)
        self.len[rid] = self.len.get(rid, 0) + len(k)

    def _joined(self, rid):
        for store in (self.k, self.v):
            if len(store[rid]) > 1:
                store[rid] = [np.concatenate(store[rid])]
        return self.k[rid][0], self.v[rid][0]

    def attend(self, rid: int, q_rows: np.ndarray, scale: float, keep=None) -> np.ndarray:
        """Attention of the last len(q_rows) positions of ``rid`` over its whole history.

        ``keep`` (indices into q_rows) restricts which rows are computed; the
        others come back as NaN.
        """
        k, v = self._joined(rid)
        n = len(q_rows)
        if keep is None:
            return attention_dense(q_rows, k, v, scale)
        out = np.full((n,) + q_rows.shape[1:], np.nan)
        for i in keep:
            # row i sees keys 0 .. L-n+i, the same as the last row of a prefix of length L-n+i+1
            L = len(k) - n + i + 1
            out[i] = attention_dense(q_rows[i:i + 1], k[:L], v[:L], scale)[0]
        return out

    def drop(self, rid: int) -> None:
        self.k.pop(rid, None)
        self.v.pop(rid, None)
        self.len.pop(rid, None)
