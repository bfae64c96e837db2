"""A small continuous-batching scheduler that produces step plans.

It exists to drive the paged-KV step through a realistic churn of arrivals,
chunked prompts, decode rows and retirements. Policy, from the pages:

* Admission needs a free slot and KV capacity for the prompt plus decode
  headroom, reserved atomically through the block pool; the deferred queue is
  strict FIFO (Lucebox, "Continuous batching: Qwen3.8-27B at 301 tok/s across
  five clients, up to 1.97x llama.cpp", §Admission and step planning are
  different decisions). The reservation here is the prompt plus the first
  decode row.
* Prompt chunks of 2048 tokens while nothing decodes, 512 while a decode batch
  runs (mlxcel manual, "Continuous batching", §Chunked prefill), shared FIFO
  across prefilling slots; prompt chunks first, decode rows after, on one
  packed axis (Lucebox §Packing unequal prompt chunks together).
* A slot stays in its prefill phase until its last chunk and decodes from the
  next step (Lucebox §Chunked prefill is a slot phase). The final chunk yields
  the first output token; each decode row one more (Tutorial 15, "Continuous
  Batching and Scheduling", §4 and §6). A request retires at the end of the
  step that produced its last token and its slot and blocks return at once
  (Lucebox §One scheduler, model-specific execution).

Budget policies (mlxcel manual, "Continuous batching", §Preemptive eviction,
§Paged KV cache and prefix sharing, §Decode headroom under a tight budget),
all off by default:

* Admission watermark F (0 <= F <= 0.5): while a decode batch runs, a request
  is admitted only if the free blocks minus F times the pool's blocks still
  cover its reservation.
* Priority preemption ("longest-first" or "lowest-priority"): when the head
  of the queue does not fit (no free slot or not enough blocks), it may evict
  an admitted request of strictly lower priority -- the one that generated
  the most tokens, or the lowest priority with most tokens breaking ties --
  and try again.
* Decode headroom: decode rows reserve the blocks they open before the step;
  if the pool cannot cover them, the eviction ladder runs: cold cached prompt
  prefixes first, prefixes adopted by waiting requests next (empty here: a
  waiting request holds no blocks), then the admitted request with the least
  progress is preempted, until the rows fit.
  Reading of "least progress": fewest generated tokens, then fewest rows in
  the cache, then the latest admitted.
* A preempted request's generated tokens are kept and its KV freed; it goes
  back into the deferred queue in arrival order and, when admitted again,
  re-prefills its prompt and the tokens it had generated (the last re-prefill
  chunk yields its next token), then decodes on. Ties between victims by
  generated tokens fall to the latest admitted.

Prompt-prefix cache (mlxcel manual, §Paged KV cache and prefix sharing), off
unless ``prefix_cache`` = C > 0 (the pool's top C slots hold the entries):

* A request whose prompt starts with a shared prefix of length p caches its
  whole blocks, c = floor(p / block) * block tokens, so no block is shared
  partly filled and no copy-on-write is ever needed.
* Donation, at the end of a step before its retirements: a request that
  prefilled the prefix itself and has reached c hands its first c / block
  blocks to a new entry by reference (``pkv_pool_adopt`` into an entry slot);
  with C entries cached, the least recently used one is dropped first.
* Admission: a head whose prefix is cached adopts the entry's blocks, is
  charged only for its suffix's blocks and prefills from position c. If the
  head lacks blocks (not a slot), cold entries -- held by the cache alone,
  other than its own -- are dropped least recently used first (ties: the
  earlier created) before priority preemption is tried.
* These cold entries are also the first rung of the decode-headroom ladder.

Slots are handed out lowest-free-first. Decode rows take new blocks inside
``pkv_plan_lower`` when their position opens one.
"""

from __future__ import annotations

import bisect
import heapq
from collections import deque
from dataclasses import dataclass

from . import binding as B


@dataclass
class _Live:
    rid: int
    slot: int
    prompt: int   # rows to prefill: the prompt, or prompt + generated tokens after a preemption
    base: int     # the request's own prompt length
    output: int
    arrival: int
    priority: int
    order: int    # admission counter (later admitted = larger)
    pos: int = 0
    decoding: bool = False
    generated: int = 0
    prefix_id: int = -1
    cached_len: int = 0   # the whole-block part of its shared prefix (0: none, or no prefix cache)
    shares: bool = False  # holds cached prefix blocks (adopted them, or donated its own)


@dataclass
class _Entry:
    """A cached prompt prefix: a pool slot holding the prefix's whole blocks by reference."""
    slot: int
    nb: int
    block0: int     # its first block (every holder of the entry holds all of its blocks)
    last_used: int
    order: int


@dataclass(frozen=True)
class PlannedRow:
    rid: int
    slot: int
    begin: int
    n: int
    prefill: bool


@dataclass
class _Waiting:
    key: tuple      # (arrival step, rid): the deferred queue's order
    rid: int
    prompt: int     # rows to prefill on admission
    base: int       # the request's own prompt length
    output: int
    priority: int
    generated: int  # tokens generated before a preemption (0 for a new request)
    prefix_id: int = -1
    cached_len: int = 0

    def __lt__(self, other):
        return self.key < other.key


class ChurnScheduler:
    def __init__(self, requests, pool: B.Pool, *, chunk_idle: int = 2048, chunk_busy: int = 512,
                 watermark: float = 0.0, preemption: str | None = None, prefix_cache: int = 0):
        if not 0.0 <= watermark <= 0.5:
            raise ValueError("watermark must be in [0, 0.5]")
        if preemption not in (None, "longest-first", "lowest-priority"):
            raise ValueError(f"unknown preemption policy {preemption!r}")
        if not 0 <= prefix_cache < pool.max_slots:
            raise ValueError("prefix_cache must leave the pool at least one request slot")
        self.pool = pool
        self.pending = deque(sorted(requests, key=lambda r: (r.arrival_step, r.rid)))
        self.queue: list[_Waiting] = []  # sorted by key
        self.live: list[_Live] = []
        # request slots first, then one slot per cache entry (the pool's top prefix_cache slots)
        self.free_slots = list(range(pool.max_slots - prefix_cache))
        heapq.heapify(self.free_slots)
        self.cache_capacity = prefix_cache
        self.cache_slots = list(range(pool.max_slots - prefix_cache, pool.max_slots))
        heapq.heapify(self.cache_slots)
        self.cache: dict[int, _Entry] = {}
        self._entries_made = 0
        # (step, event, prefix id): "donate", "adopt", "drop-capacity", "drop-admission", "drop-headroom"
        self.cache_events: list[tuple] = []
        self.chunk_idle, self.chunk_busy = chunk_idle, chunk_busy
        self.watermark, self.preemption = watermark, preemption
        self.step_index = 0
        self.admitted = 0
        self.preempted: list[int] = []  # request IDs, in preemption order
        self.preempt_reasons: list[str] = []  # "priority" or "headroom", one per preemption

    # ---- helpers ------------------------------------------------------------
    def _free_blocks(self) -> int:
        return self.pool.stats().free_blocks

    def _cached_len(self, prefix_id: int, prefix_len: int) -> int:
        bs = self.pool.block_size
        return (prefix_len // bs) * bs if self.cache_capacity > 0 and prefix_id >= 0 else 0

    def _drop(self, e_pid: int, why: str) -> None:
        e = self.cache.pop(e_pid)
        self.pool.release(e.slot)
        heapq.heappush(self.cache_slots, e.slot)
        self.cache_events.append((self.step_index, "drop-" + why, e_pid))

    def _cold(self, spare: int | None = None) -> list[int]:
        """Prefix IDs of entries whose blocks only the cache holds, least recently used first."""
        cold = [(e.last_used, e.order, pid) for pid, e in self.cache.items()
                if pid != spare and self.pool.block_refs(e.block0) == 1]
        return [pid for _, _, pid in sorted(cold)]

    def _preempt(self, r: _Live, reason: str, hold: list | None = None) -> None:
        """Release r; it waits again in arrival order (in ``hold`` until the request that evicted it is in)."""
        self.pool.release(r.slot)
        heapq.heappush(self.free_slots, r.slot)
        self.live.remove(r)
        # re-prefill the prompt and every generated token; keep the count of generated tokens
        w = _Waiting((r.arrival, r.rid), r.rid, r.base + r.generated, r.base, r.output, r.priority, r.generated,
                     r.prefix_id, r.cached_len)
        if hold is None:
            bisect.insort(self.queue, w)
        else:
            hold.append(w)
        self.preempted.append(r.rid)
        self.preempt_reasons.append(reason)

    def _priority_victim(self, priority: int):
        cands = [r for r in self.live if r.priority < priority]
        if not cands:
            return None
        if self.preemption == "lowest-priority":
            return min(cands, key=lambda r: (r.priority, -r.generated, -r.order))
        return max(cands, key=lambda r: (r.generated, r.order))

    def _decode_blocks_needed(self) -> int:
        bs = self.pool.block_size
        return sum(1 for r in self.live if r.decoding and r.pos // bs >= self.pool.slot_blocks(r.slot))

    # ---- one step -------------------------------------------------------------
    def plan(self) -> list[PlannedRow]:
        s = self.step_index
        bs = self.pool.block_size
        while self.pending and self.pending[0].arrival_step <= s:
            q = self.pending.popleft()
            bisect.insort(self.queue, _Waiting((q.arrival_step, q.rid), q.rid, q.prompt_len, q.prompt_len,
                                               q.output_len, q.priority, 0, q.prefix_id,
                                               self._cached_len(q.prefix_id, q.prefix_len)))
        hold: list[_Waiting] = []  # evicted for the current head: they queue up behind it
        while self.queue:
            head = self.queue[0]
            e = self.cache.get(head.prefix_id) if head.cached_len > 0 else None
            need = -(-(head.prompt + 1) // bs) - (e.nb if e else 0)
            mark = self.watermark * self.pool.num_blocks if any(r.decoding for r in self.live) else 0.0
            if not self.free_slots or self._free_blocks() - need < mark:
                cold = self._cold(spare=head.prefix_id if e else None) if self.free_slots else []
                if cold:  # first rung: a cold cached prefix
                    self._drop(cold[0], "admission")
                    continue
                victim = self._priority_victim(head.priority) if self.preemption else None
                if victim is None:
                    break  # strict FIFO: the head waits, nobody behind it jumps ahead
                self._preempt(victim, "priority", hold)
                continue
            slot = self.free_slots[0]
            if e is not None:  # adopt the cached prefix; prefill starts after it
                rc = self.pool.adopt(slot, e.slot, head.cached_len, head.prompt + 1)
                if rc != B.PKV_OK:
                    raise B.PkvError(rc, "pkv_pool_adopt")
                e.last_used = s
                self.cache_events.append((s, "adopt", head.prefix_id))
            else:
                rc = self.pool.admit(slot, head.prompt + 1)
                if rc != B.PKV_OK:
                    raise B.PkvError(rc, "pkv_pool_admit")
            heapq.heappop(self.free_slots)
            self.queue.pop(0)
            for w in hold:
                bisect.insort(self.queue, w)
            hold.clear()
            r = _Live(head.rid, slot, head.prompt, head.base, head.output, head.key[0], head.priority, self.admitted)
            r.generated = head.generated
            r.prefix_id, r.cached_len = head.prefix_id, head.cached_len
            if e is not None:
                r.pos, r.shares = head.cached_len, True
            self.admitted += 1
            self.live.append(r)
        for w in hold:  # the head did not fit even after every eviction it could make
            bisect.insort(self.queue, w)
        # decode headroom: blocks the decode rows open must be free before the step
        while self._decode_blocks_needed() > self._free_blocks():
            cold = self._cold()
            if cold:  # first rung: a cold cached prefix; no waiting request holds blocks (second rung)
                self._drop(cold[0], "headroom")
                continue
            victim = min(self.live, key=lambda r: (r.generated, r.pos, -r.order))
            self._preempt(victim, "headroom")
        budget = self.chunk_busy if any(r.decoding for r in self.live) else self.chunk_idle
        rows: list[PlannedRow] = []
        for r in self.live:
            if budget == 0:
                break
            if not r.decoding and r.pos < r.prompt:
                take = min(r.prompt - r.pos, budget)
                rows.append(PlannedRow(r.rid, r.slot, r.pos, take, True))
                budget -= take
        rows.extend(PlannedRow(r.rid, r.slot, r.pos, 1, False) for r in self.live if r.decoding)
        return rows

    def commit(self, rows: list[PlannedRow]) -> list[int]:
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
        # donations, before this step's retirements: the prefix's whole blocks go to a cache entry
        for r in self.live:
            if r.cached_len > 0 and not r.shares and r.pos >= r.cached_len and r.prefix_id not in self.cache:
                if len(self.cache) >= self.cache_capacity:
                    lru = min(self.cache, key=lambda pid: (self.cache[pid].last_used, self.cache[pid].order))
                    self._drop(lru, "capacity")
                slot = heapq.heappop(self.cache_slots)
                rc = self.pool.adopt(slot, r.slot, r.cached_len, r.cached_len)
                if rc != B.PKV_OK:
                    raise B.PkvError(rc, "pkv_pool_adopt")
                block0 = int(self.pool.block_tables()[slot][0])
                self.cache[r.prefix_id] = _Entry(slot, r.cached_len // self.pool.block_size, block0,
                                                 self.step_index, self._entries_made)
                self._entries_made += 1
                r.shares = True
                self.cache_events.append((self.step_index, "donate", r.prefix_id))
        for rid in done:
            r = by_rid[rid]
            self.pool.release(r.slot)
            heapq.heappush(self.free_slots, r.slot)
            self.live.remove(r)
        self.step_index += 1
        return done
