"""Admission and step-composition policy, in plain Python (oracle).

TEST INFRASTRUCTURE ONLY -- see the package docstring for who may import it.

Source: "20.3 服务、批处理与流式", section 20.3.2 批处理, the
Forma batch mode and its scaled illustration:
  * all slots share one pool of fixed-size KV blocks (32 positions; the
    illustration scales this to 4), allocated on demand;
  * admitting a request whenever a slot is free can deadlock: every slot
    busy, the pool empty, no sequence able to grow, so nothing finishes and
    nothing is freed.  Admission therefore reserves blocks for the prompt
    *and* for part of the answer, so that an admitted request can finish;
  * each step first schedules the prefill chunks of sequences that have no
    first token yet (512 tokens per chunk; 8 in the illustration), then one
    row for every decoding sequence; rows that do not fit wait for the next
    step and are not evicted;
  * at most a fixed number of rows per step (12 in the illustration);
  * the request queue is served first-come first-served (section 20.3.4).
Page "大模型推理为什么需要 Continuous Batching", section 2.2 and 3.3: after each
step finished sequences leave and waiting requests fill the freed slots.

Readings where the pages leave the step open (listed in the design notes):
  R7  chunk = min(chunk, prompt left, rows left); prefills in admission
      order; decode rows ordered by (steps waited desc, admission order).
  R8  lowest free slot; blocks from a min-heap (lowest id first).
  R9  admit the queue head iff a slot is free and
          free_blocks - sum(outstanding reservations) >= blocks(prompt +
          min(max_tokens, answer_budget)),
      outstanding = reserved - allocated (>= 0).  Growth inside a
      reservation always succeeds; growth beyond it takes an unreserved free
      block or the row waits, and admission freezes while any row waits for
      a block.  If every running sequence is stuck, the youngest is stopped
      with reason LENGTH_FALLBACK (counted; never happens with an ample pool).
  R10 strict FCFS: a head that does not fit blocks the queue.
  R11 no EOS: a request finishes when it has max_tokens generated tokens.
  Positions: prompt tokens occupy 0..P-1; the last prefill row samples the
  first generated token; decode row k feeds generated token k at position
  P + k.  A request needs P + max_tokens - 1 positions.

``reserve_answer=False`` gives the free-slot-only admission the page warns
about; ``stall_fallback=False`` makes plan() report a deadlock instead of
stopping a sequence.

Overload and backpressure, same page, section 20.3.4 背压与取消 (each is off
when its config value is 0):
  * the admission queue is bounded (Forma: 8 waiters per slot); a request
    that arrives to a full queue is refused at once ("busy, retry later");
  * a request that has waited longer than the wait budget (Forma: 30 s) is
    turned away -- an outcome distinct from the client cancelling;
  * tokens go to each request through a bounded buffer that the client
    drains; a send that finds the buffer full is not made, the client is
    judged to be lagging and its request is cancelled, so a slow client
    never stalls the batch (the page's two-stream program: buffer 2, the
    slow stream is cancelled at step 3 holding 2 tokens);
  * a client that goes away stops its generation at once and gives back its
    KV blocks.
Readings: R30 a lagging request keeps the tokens it had delivered; the one
that did not fit is dropped.  R31 the queue bound counts requests not yet
admitted.  R32 expiry is checked at each plan, before admission, with a
caller-driven clock in milliseconds (wait > budget).  R33 an abort of a
request whose step is in flight (planned, not committed) takes effect at
that commit, which drops its token, since the step still writes its blocks.

A second composition policy (``policy="albatross"``), from page "RWKV Runner
Albatross 后端", section 连续批处理：Worker 主循环 (the worker's main loop):
  * the task pool is filled from the queue up to the batch size, but with
    at most max_prefill_count = max(int(batch_size * 0.125), 1) requests in
    prefill at once, so prefill cannot crowd out decoding;
  * a prompt shorter than min_forward_seq_len = 10 tokens is prefilled one
    token per step alongside the decode rows, instead of by a sequence
    forward;
  * longer prompts are prefilled by sequence forwards, paced by
    decode_prefill_ratio = 5: one sequence forward after about every 5
    decode rounds, so long prefills fill the gaps between decode rounds.
Readings: R34 the batch size is max_slots (the page's one spare slot is for
its in-place state swaps, which block tables make unnecessary); admission
keeps the block reservation of R9 and FCFS.  R35 a sequence step gives every
long prompt in prefill one chunk and also carries the decode and one-token
rows (the step is mixed); it comes when prefill_every steps with other rows
have passed since the last one, or at once when no other row exists.
"""
from __future__ import annotations

import dataclasses
import heapq
from collections import deque

FINISH_LENGTH = 1            # reached max_tokens
FINISH_LENGTH_FALLBACK = 2   # stopped because every running sequence was stuck
FINISH_ABORTED = 3           # the client went away
FINISH_TIMEOUT = 4           # waited longer than the queue's wait budget
FINISH_LAGGING = 5           # delivery buffer full: slow client cancelled


class Deadlock(Exception):
    """No running sequence can make progress and no fallback is allowed."""


class PoolTooSmall(Exception):
    """The request can never be admitted."""


class Busy(Exception):
    """The admission queue is full; the client should retry later."""


def blocks_for(positions: int, block_size: int) -> int:
    return -(-positions // block_size)


@dataclasses.dataclass
class SchedConfig:
    n_blocks: int
    block_size: int = 32
    max_slots: int = 64
    max_rows: int = 2048
    chunk: int = 512
    answer_budget: int = 128
    max_blocks_per_seq: int = 1024
    reserve_answer: bool = True
    stall_fallback: bool = True
    queue_per_slot: int = 0      # waiting requests per slot (0: unbounded)
    queue_timeout_ms: int = 0    # wait budget (0: none)
    out_buffer: int = 0          # undelivered tokens per request (0: unbounded, untracked)
    policy: str = "forma"        # or "albatross"
    max_prefill: int = 0         # albatross: 0 -> max(int(0.125 * max_slots), 1)
    prefill_every: int = 0       # albatross: 0 -> 5 (decode_prefill_ratio)
    short_prompt: int = 0        # albatross: 0 -> 10 (min_forward_seq_len)


@dataclasses.dataclass
class Request:
    id: int
    prompt: list
    max_tokens: int
    sampling: object = None
    slot: int = -1
    blocks: list = dataclasses.field(default_factory=list)
    reserved: int = 0
    n_prefilled: int = 0
    generated: list = dataclasses.field(default_factory=list)
    waited: int = 0
    block_wait: bool = False
    admit_seq: int = -1
    pending_prefill: int = 0
    arrival_ms: int = 0
    aborted: bool = False
    outbox: deque = dataclasses.field(default_factory=deque)


@dataclasses.dataclass
class Plan:
    rows: list            # (slot, token, pos, is_prefill, sample)
    sampled: list         # (request id, token_index) per sampled row, in row order
    block_tables: dict    # slot -> list of physical block ids (logical order)
    resets: list          # slots whose penalty counters start at zero
    stopped: list         # (request id, reason) stopped by the stall fallback


class Scheduler:
    def __init__(self, cfg: SchedConfig):
        self.cfg = cfg
        self.free = list(range(cfg.n_blocks))
        heapq.heapify(self.free)
        self.slots = [None] * cfg.max_slots
        self.waiting = deque()
        self.running = []           # admission order
        self.finished = {}          # id -> (reason, generated)
        self._admit_counter = 0
        self._last_plan = None
        self.n_fallback = 0
        self.now_ms = 0
        self.side_finished = []     # (id, reason, n_tokens) finished outside a commit
        self.outboxes = {}          # id -> deque of undelivered tokens of finished requests
        self.counts = dict(rejected_busy=0, timed_out=0, aborted=0, lagging=0)
        self.seq_countdown = 0      # albatross: steps left before the next sequence step
        c = cfg
        self.alb = c.policy == "albatross"
        self.max_prefill = c.max_prefill or max(int(c.max_slots * 0.125), 1)
        self.prefill_every = c.prefill_every or 5
        self.short_prompt = c.short_prompt or 10

    # -- helpers -------------------------------------------------------
    def _need(self, req: Request) -> int:
        c = self.cfg
        if not c.reserve_answer:
            return 0
        return blocks_for(len(req.prompt) + min(req.max_tokens, c.answer_budget), c.block_size)

    def _outstanding(self) -> int:
        return sum(max(0, r.reserved - len(r.blocks)) for r in self.running)

    def _grow(self, req: Request) -> bool:
        """Give req one more block; False if none may be taken."""
        if not self.free:
            return False
        if len(req.blocks) < req.reserved:
            req.blocks.append(heapq.heappop(self.free))
            return True
        if len(self.free) - self._outstanding() > 0:
            req.blocks.append(heapq.heappop(self.free))
            return True
        return False

    def _release(self, req: Request, reason: int) -> None:
        for b in req.blocks:
            heapq.heappush(self.free, b)
        req.blocks = []
        self.slots[req.slot] = None
        self.running.remove(req)
        self.finished[req.id] = (reason, list(req.generated))
        self.outboxes[req.id] = req.outbox

    # -- public API ----------------------------------------------------
    def submit(self, req: Request) -> None:
        c = self.cfg
        if len(req.prompt) < 1 or req.max_tokens < 1:
            raise ValueError("empty prompt or max_tokens < 1")
        total = len(req.prompt) + req.max_tokens - 1
        if blocks_for(total, c.block_size) > c.max_blocks_per_seq:
            raise PoolTooSmall("request longer than max_blocks_per_seq")
        first = blocks_for(len(req.prompt) + min(req.max_tokens, c.answer_budget), c.block_size)
        if first > c.n_blocks:
            raise PoolTooSmall("request can never fit the pool")
        if c.queue_per_slot and len(self.waiting) >= c.queue_per_slot * c.max_slots:
            self.counts["rejected_busy"] += 1
            raise Busy("admission queue full")
        req.arrival_ms = self.now_ms
        self.waiting.append(req)

    def set_time(self, now_ms: int) -> None:
        if now_ms < self.now_ms:
            raise ValueError("the clock must not go backwards")
        self.now_ms = now_ms

    def _expire(self) -> None:
        """Waiters past the wait budget leave the queue (R32)."""
        c = self.cfg
        if not c.queue_timeout_ms:
            return
        keep = deque()
        for r in self.waiting:
            if self.now_ms - r.arrival_ms > c.queue_timeout_ms:
                self.finished[r.id] = (FINISH_TIMEOUT, [])
                self.outboxes[r.id] = deque()
                self.side_finished.append((r.id, FINISH_TIMEOUT, 0))
                self.counts["timed_out"] += 1
            else:
                keep.append(r)
        self.waiting = keep

    def abort(self, rid: int) -> None:
        """The client went away: stop now, or at the commit of the step in flight (R33)."""
        for r in list(self.waiting):
            if r.id == rid:
                self.waiting.remove(r)
                self.finished[rid] = (FINISH_ABORTED, [])
                self.outboxes[rid] = deque()
                self.side_finished.append((rid, FINISH_ABORTED, 0))
                self.counts["aborted"] += 1
                return
        for r in self.running:
            if r.id == rid:
                if r.aborted:
                    raise ValueError("already aborted")
                if self._last_plan is not None:
                    r.aborted = True
                    return
                self.side_finished.append((rid, FINISH_ABORTED, len(r.generated)))
                self.counts["aborted"] += 1
                self._release(r, FINISH_ABORTED)
                return
        raise ValueError("unknown or finished request")

    def read(self, rid: int, cap: int = 1 << 30) -> list:
        """The client drains up to cap undelivered tokens, oldest first."""
        box = None
        for r in self.running:
            if r.id == rid:
                box = r.outbox
        if box is None:
            box = self.outboxes.get(rid)
        if box is None:
            if any(r.id == rid for r in self.waiting):
                return []
            raise ValueError("unknown request")
        out = []
        while box and len(out) < cap:
            out.append(box.popleft())
        return out

    def take_finished(self) -> list:
        out, self.side_finished = self.side_finished, []
        return out

    def _admit(self, resets: list) -> None:
        """Admission (R9, R10): FCFS; frozen while a row waits for a block."""
        c = self.cfg
        if any(r.block_wait for r in self.running):
            return
        prefilling = sum(1 for r in self.running if r.n_prefilled < len(r.prompt))
        while self.waiting and None in self.slots:
            if self.alb and prefilling >= self.max_prefill:
                return
            head = self.waiting[0]
            need = self._need(head)
            if c.reserve_answer and len(self.free) - self._outstanding() < need:
                return
            self.waiting.popleft()
            head.slot = self.slots.index(None)
            self.slots[head.slot] = head
            head.reserved = need
            head.admit_seq = self._admit_counter
            self._admit_counter += 1
            self.running.append(head)
            resets.append(head.slot)
            prefilling += 1

    def _compose(self):
        """Rows of one step: prefill chunks first, then one row per decoder.

        Returns (rows, sampled, waits) where waits lists (request, for_block)
        of rows that did not fit; block grants are applied as rows are made.
        """
        c = self.cfg
        rows, sampled, waits = [], [], []
        budget = c.max_rows
        prefilling = set()
        for r in self.running:
            r.pending_prefill = 0
        seq_step = False
        if self.alb:
            other = any((r.n_prefilled < len(r.prompt) and len(r.prompt) < self.short_prompt) or
                        (r.n_prefilled == len(r.prompt) and 0 < len(r.generated) < r.max_tokens)
                        for r in self.running)
            any_seq = any(r.n_prefilled < len(r.prompt) and len(r.prompt) >= self.short_prompt
                          for r in self.running)
            seq_step = any_seq and (self.seq_countdown <= 0 or not other)
        self._seq_step = seq_step
        for r in self.running:                                   # prefill chunks
            if r.n_prefilled >= len(r.prompt):
                continue
            take = c.chunk
            if self.alb:
                if len(r.prompt) < self.short_prompt:
                    take = 1                                     # one token per step
                elif not seq_step:
                    continue                                     # waits for a sequence step
            if budget == 0:
                waits.append((r, False))
                continue
            n = min(take, len(r.prompt) - r.n_prefilled, budget)
            while len(r.blocks) * c.block_size < r.n_prefilled + n and self._grow(r):
                pass
            n = min(n, len(r.blocks) * c.block_size - r.n_prefilled)
            if n <= 0:
                waits.append((r, True))
                continue
            done = r.n_prefilled + n == len(r.prompt)
            for i in range(n):
                p = r.n_prefilled + i
                smp = 1 if (done and i == n - 1) else 0
                rows.append((r.slot, r.prompt[p], p, 1, smp))
                if smp:
                    sampled.append((r.id, 0))
            r.pending_prefill = n
            prefilling.add(r.id)
            budget -= n
        decoding = [r for r in self.running
                    if r.n_prefilled == len(r.prompt) and r.id not in prefilling
                    and 0 < len(r.generated) < r.max_tokens]
        decoding.sort(key=lambda r: (-r.waited, r.admit_seq))
        for r in decoding:                                       # one row each
            pos = len(r.prompt) + len(r.generated) - 1
            if budget == 0:
                waits.append((r, False))
                continue
            if pos >= len(r.blocks) * c.block_size and not self._grow(r):
                waits.append((r, True))
                continue
            rows.append((r.slot, r.generated[-1], pos, 0, 1))
            sampled.append((r.id, len(r.generated)))
            budget -= 1
        return rows, sampled, waits

    def plan(self) -> Plan:
        c = self.cfg
        resets, stopped = [], []
        self._expire()
        self._admit(resets)
        while True:
            rows, sampled, waits = self._compose()
            if rows or not self.running:
                break
            if not c.stall_fallback:
                raise Deadlock("every running sequence is stuck")
            young = max(self.running, key=lambda r: r.admit_seq)   # R9 fallback
            stopped.append((young.id, FINISH_LENGTH_FALLBACK))
            self.n_fallback += 1
            self._release(young, FINISH_LENGTH_FALLBACK)
        if self.alb and rows:
            if self._seq_step:
                self.seq_countdown = self.prefill_every
            else:
                self.seq_countdown = max(self.seq_countdown - 1, 0)
        waiting_ids = {id(r) for r, _ in waits}
        for r in self.running:
            if id(r) in waiting_ids:
                r.waited += 1
            else:
                r.waited = 0
            r.block_wait = False
        for r, for_block in waits:
            r.block_wait = r.block_wait or for_block
        tables = {r.slot: list(r.blocks) for r in self.running}
        plan = Plan(rows, sampled, tables, resets, stopped)
        self._last_plan = plan
        return plan

    def commit(self, tokens) -> list:
        """Feed the sampled tokens of the last plan (row order).

        Returns [(request id, reason)] of requests finished by this commit.
        """
        plan = self._last_plan
        if plan is None:
            raise RuntimeError("commit without plan")
        if len(tokens) != len(plan.sampled):
            raise ValueError("token count does not match the plan")
        ob = self.cfg.out_buffer
        by_id = {r.id: r for r in self.running}
        for r in self.running:
            r.n_prefilled += r.pending_prefill
            r.pending_prefill = 0
        lagging = set()
        for (rid, _), t in zip(plan.sampled, tokens):      # delivery, row order
            r = by_id[rid]
            if r.aborted or rid in lagging:
                continue
            if ob and len(r.outbox) >= ob:                  # buffer full: cancel (R30)
                lagging.add(rid)
                continue
            r.generated.append(int(t))
            if ob:
                r.outbox.append(int(t))
        done = []
        for r in list(self.running):
            if r.aborted:
                why = FINISH_ABORTED
                self.counts["aborted"] += 1
            elif r.id in lagging:
                why = FINISH_LAGGING
                self.counts["lagging"] += 1
            elif len(r.generated) >= r.max_tokens:
                why = FINISH_LENGTH
            else:
                continue
            self._release(r, why)
            done.append((r.id, why))
        self._last_plan = None
        return done

    def stats(self) -> dict:
        return dict(running=len(self.running), waiting=len(self.waiting),
                    free_blocks=len(self.free), outstanding=self._outstanding(),
                    allocated=sum(len(r.blocks) for r in self.running),
                    reserved=sum(r.reserved for r in self.running),
                    fallback_stops=self.n_fallback, **self.counts)
