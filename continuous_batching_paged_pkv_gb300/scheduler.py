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

Slots are handed out lowest-free-first. Decode rows take new blocks inside
``pkv_plan_lower`` when their position opens one.
"""

from __future__ import annotations

import heapq
from collections import deque
from dataclasses import dataclass

from . import binding as B


@dataclass
class _Live:
    rid: int
    slot: int
    prompt: int
    output: int
    pos: int = 0
    decoding: bool = False
    generated: int = 0


@dataclass(frozen=True)
class PlannedRow:
    rid: int
    slot: int
    begin: int
    n: int
    prefill: bool


class ChurnScheduler:
    def __init__(self, requests, pool: B.Pool, *, chunk_idle: int = 2048, chunk_busy: int = 512):
        self.pool = pool
        self.pending = deque(sorted(requests, key=lambda r: (r.arrival_step, r.rid)))
        self.queue: deque = deque()
        self.live: list[_Live] = []
        self.free_slots = list(range(pool.max_slots))
        heapq.heapify(self.free_slots)
        self.chunk_idle, self.chunk_busy = chunk_idle, chunk_busy
        self.step_index = 0

    def plan(self) -> list[PlannedRow]:
        s = self.step_index
        while self.pending and self.pending[0].arrival_step <= s:
            self.queue.append(self.pending.popleft())
        while self.queue and self.free_slots:
            head = self.queue[0]
            slot = self.free_slots[0]
            rc = self.pool.admit(slot, head.prompt_len + 1)
            if rc == B.PKV_ERR_NO_BLOCKS:
                break  # strict FIFO
            if rc != B.PKV_OK:
                raise B.PkvError(rc, "pkv_pool_admit")
            heapq.heappop(self.free_slots)
            self.queue.popleft()
            self.live.append(_Live(head.rid, slot, head.prompt_len, head.output_len))
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
                    r.generated = 1
            else:
                r.generated += 1
            if r.pos >= r.prompt and r.generated >= r.output:
                done.append(r.rid)
        for rid in done:
            r = by_rid[rid]
            self.pool.release(r.slot)
            heapq.heappush(self.free_slots, r.slot)
            self.live.remove(r)
        self.step_index += 1
        return done
