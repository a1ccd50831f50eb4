"""Pins for the overload and backpressure rules of the scheduler simulator
("20.3 服务、批处理与流式", section 20.3.4 背压与取消), CPU only:

* the page's two-stream program (bounded delivery buffer of 2 tokens, one
  client never reads): its printed outcome, stored in tests/golden;
* the bounded admission queue (waiters per slot) and the wait budget, and
  that a timeout and a client cancel are different outcomes;
* aborts while queued, between steps and with the step in flight: the KV
  blocks come back and the other requests carry on;
* invariants on random traces with arrivals over time, aborts and slow
  readers: pool accounting, every request ending exactly once.
"""
import os
import random

import pytest

from oracle import sched_sim as ss

GOLD = os.path.join(os.path.dirname(__file__), "golden", "backpressure_two_streams.txt")


def golden():
    remaining, cancelled, buf = {}, None, None
    for line in open(GOLD):
        f = line.split()
        if not f or f[0].startswith("#"):
            continue
        if f[0] == "buffer":
            buf = int(f[1])
        elif f[0] == "remaining":
            remaining[int(f[1])] = int(f[2])
        elif f[0] == "cancelled":
            cancelled = (int(f[1]), int(f[2]))
    return buf, remaining, cancelled


def test_two_stream_program_from_the_page():
    buf, remaining, (cancel_step, held) = golden()
    s = ss.Scheduler(ss.SchedConfig(n_blocks=64, block_size=4, max_slots=4, max_rows=16, chunk=8,
                                    answer_budget=16, max_blocks_per_seq=64, out_buffer=buf))
    FAST, SLOW = 0, 1
    s.submit(ss.Request(FAST, [5], 50))
    s.submit(ss.Request(SLOW, [6], 50))
    for step in range(1, max(remaining) + 1):
        p = s.plan()
        done = s.commit([100 * step + i for i in range(len(p.sampled))])
        if step == cancel_step:
            assert done == [(SLOW, ss.FINISH_LAGGING)]
            assert s.read(SLOW) == [101, 201][:held] and len(s.finished[SLOW][1]) == held
        else:
            assert done == []
        assert s.read(FAST, 1) == [100 * step]   # the fast client reads one token per step
        assert len(s.running) == remaining[step], step
    assert s.counts["lagging"] == 1
    assert s.read(FAST) == []                # it kept up: nothing left over


def test_admission_queue_bound_and_busy():
    s = ss.Scheduler(ss.SchedConfig(n_blocks=400, block_size=4, max_slots=2, max_rows=64, chunk=8,
                                    answer_budget=16, max_blocks_per_seq=64, queue_per_slot=8))
    for i in range(16):                       # 8 waiters per slot, 2 slots
        s.submit(ss.Request(i, [1, 2, 3], 4))
    with pytest.raises(ss.Busy):
        s.submit(ss.Request(16, [1, 2, 3], 4))
    assert s.counts["rejected_busy"] == 1
    s.plan()                                  # two admitted: two places free in the queue
    s.submit(ss.Request(16, [1, 2, 3], 4))
    s.submit(ss.Request(17, [1, 2, 3], 4))
    with pytest.raises(ss.Busy):
        s.submit(ss.Request(18, [1, 2, 3], 4))


def test_wait_budget_is_distinct_from_cancel():
    s = ss.Scheduler(ss.SchedConfig(n_blocks=400, block_size=4, max_slots=1, max_rows=64, chunk=8,
                                    answer_budget=16, max_blocks_per_seq=64, queue_timeout_ms=30000))
    s.submit(ss.Request(0, [1, 2], 100))     # holds the only slot
    s.plan(); s.commit([7])
    s.set_time(1000)
    s.submit(ss.Request(1, [3], 4))          # arrives at t = 1 s
    s.submit(ss.Request(2, [4], 4))
    s.set_time(31000)                        # waited exactly 30 s: not more than the budget
    s.plan(); s.commit([8])
    assert s.take_finished() == []
    s.abort(2)                               # the client of request 2 leaves
    s.set_time(31001)
    s.plan(); s.commit([9])
    assert s.take_finished() == [(2, ss.FINISH_ABORTED, 0), (1, ss.FINISH_TIMEOUT, 0)]
    assert s.finished[1][0] == ss.FINISH_TIMEOUT and s.finished[2][0] == ss.FINISH_ABORTED
    assert s.counts["timed_out"] == 1 and s.counts["aborted"] == 1
    with pytest.raises(ValueError):
        s.set_time(30000)                    # the clock does not go back


def test_abort_returns_blocks_at_every_stage():
    cfg = ss.SchedConfig(n_blocks=20, block_size=4, max_slots=2, max_rows=12, chunk=8, answer_budget=8,
                         max_blocks_per_seq=64)
    s = ss.Scheduler(cfg)
    s.submit(ss.Request(0, list(range(20)), 6))          # long prompt: several chunks
    s.submit(ss.Request(1, [1, 2, 3], 6))
    s.submit(ss.Request(2, [4, 5], 6))                   # waits for a slot
    p = s.plan()                                         # 0: first chunk; 1: whole prompt
    s.abort(0)                                           # mid-prefill, step in flight
    assert any(r.id == 0 for r in s.running)             # its blocks still belong to the step
    done = s.commit([11] * len(p.sampled))
    assert (0, ss.FINISH_ABORTED) in done
    assert s.finished[0] == (ss.FINISH_ABORTED, [])      # no token reached the client
    p = s.plan()                                         # request 2 takes the freed slot
    assert p.resets == [0]
    s.commit([12] * len(p.sampled))
    s.abort(1)                                           # between steps: freed at once
    assert s.take_finished() == [(1, ss.FINISH_ABORTED, 2)]
    assert s.stats()["allocated"] == len(s.running[0].blocks)
    while s.running:
        p = s.plan()
        s.commit([13] * len(p.sampled))
    assert s.finished[2][0] == ss.FINISH_LENGTH and len(s.finished[2][1]) == 6
    assert len(s.free) == cfg.n_blocks
    with pytest.raises(ValueError):
        s.abort(2)                                       # already finished


def drive(s, rng, reqs, abort_p=0.03, slow=frozenset(), max_steps=20000):
    """Arrivals over time, random aborts, clients that read (or not)."""
    pending = list(reqs)                                  # (arrival_ms, id, prompt, max_tokens)
    t, steps, outcome = 0, 0, {}
    while pending or s.running or s.waiting:
        t += rng.choice([5, 20, 200])
        s.set_time(t)
        while pending and pending[0][0] <= t:
            _, rid, prompt, mt = pending.pop(0)
            try:
                s.submit(ss.Request(rid, prompt, mt))
            except ss.Busy:
                outcome[rid] = "busy"
        live = [r.id for r in s.running] + [r.id for r in s.waiting]
        if live and rng.random() < abort_p:
            s.abort(rng.choice(live))
        p = s.plan()
        in_flight = [r.id for r in s.running if not r.aborted]
        if in_flight and rng.random() < abort_p:
            s.abort(rng.choice(in_flight))                # takes effect at this commit
        for rid, why in s.commit([rng.randrange(1000) for _ in p.sampled]):
            assert rid not in outcome
            outcome[rid] = why
        for rid, why, _ in s.take_finished():
            assert rid not in outcome
            outcome[rid] = why
        for r in s.running:
            if r.id not in slow:
                s.read(r.id, 2)
        st = s.stats()
        assert st["allocated"] + st["outstanding"] <= s.cfg.n_blocks
        steps += 1
        assert steps < max_steps
    return outcome


@pytest.mark.parametrize("seed", range(5))
def test_random_traces_with_overload_and_aborts(seed):
    rng = random.Random(seed)
    cfg = ss.SchedConfig(n_blocks=rng.choice([40, 200]), block_size=4, max_slots=rng.choice([2, 6]),
                         max_rows=rng.choice([16, 48]), chunk=8, answer_budget=16, max_blocks_per_seq=200,
                         queue_per_slot=rng.choice([2, 8]), queue_timeout_ms=rng.choice([500, 3000]),
                         out_buffer=rng.choice([2, 4]))
    s = ss.Scheduler(cfg)
    t, reqs = 0, []
    for i in range(60):
        t += rng.choice([0, 10, 50])
        reqs.append((t, i, [rng.randrange(100) for _ in range(rng.randint(1, 30))], rng.randint(1, 30)))
    slow = frozenset(rng.sample(range(60), 6))
    outcome = drive(s, rng, reqs, slow=slow)
    assert sorted(outcome) == list(range(60))            # every request ended exactly once
    assert len(s.free) == cfg.n_blocks and not s.running and not s.waiting
    for rid, why in outcome.items():
        if why == ss.FINISH_LENGTH:
            assert len(s.finished[rid][1]) == reqs[rid][3]
        if why == ss.FINISH_LAGGING:
            assert len(s.finished[rid][1]) >= cfg.out_buffer
