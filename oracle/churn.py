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
  free; otherwise admitted requests are preempted, least progress first
  (reading: fewest generated tokens, then fewest cached rows, then latest
  admitted), until they are. (The pages' earlier rungs, cold cached prefixes
  and prefixes adopted by waiting requests, do not exist in this replay.)
* A preempted request frees its slot and blocks, keeps its generated-token
  count, and waits again in arrival order; once admitted it prefills its
  prompt plus the tokens it had generated, the last chunk yielding one more
  token, then decodes.
"""

from __future__ import annotations

from collections import deque
from dataclasses import dataclass

import numpy as np

from . import attention_dense


@dataclass
class _Live:
    rid: int
    prompt: int
    output: int
    pos: int = 0
    decoding: bool = False
    generated: int = 0
    blocks: int = 0
    own_prompt: int = 0
    arrival: int = 0
    priority: int = 0
    admitted_as: int = 0


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
                 preemption: str | None = None):
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

    def _evict(self, r: _Live, reason: str, held=None) -> None:
        """Free r's slot and blocks; it waits again (in `held` until the request that evicted it is in)."""
        self.live.remove(r)
        self.free_slots += 1
        self.free_blocks += r.blocks
        entry = (r.arrival, r.rid, r.own_prompt + r.generated, r.own_prompt, r.output, r.priority, r.generated)
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
            self.queue.append((q.arrival_step, q.rid, q.prompt_len, q.prompt_len, q.output_len,
                               getattr(q, "priority", 0), 0))
            self.queue.sort()
        held: list[tuple] = []  # evicted for the current head; they wait behind it
        while self.queue:
            arrival, rid, rows_to_fill, own, output, prio, gen = self.queue[0]
            need = _ceil_div(rows_to_fill + 1, self.bs)
            floor = self.watermark * self.num_blocks if any(r.decoding for r in self.live) else 0.0
            if self.free_slots == 0 or self.free_blocks - need < floor:
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
            self.live.append(_Live(rid, rows_to_fill, output, generated=gen, blocks=need, own_prompt=own,
                                   arrival=arrival, priority=prio, admitted_as=self._admissions))
            self._admissions += 1
        if held:  # the head still did not fit after every eviction it could make
            self.queue.extend(held)
            self.queue.sort()
        # decode headroom
        while True:
            opening = sum(1 for r in self.live if r.decoding and r.pos // self.bs >= r.blocks)
            if opening <= self.free_blocks:
                break
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
                if r.pos // self.bs >= r.blocks:
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
        for rid in done:
            r = by_rid[rid]
            self.live.remove(r)
            self.free_slots += 1
            self.free_blocks += r.blocks
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
