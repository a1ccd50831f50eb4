"""Pins for the scheduler simulator (CPU only).

* a plan worked out by hand on the scaled constants of the page's
  illustration (4 slots, 4 positions per block, 8-token chunks, 12 rows);
* the deadlock the page describes: admitting whenever a slot is free
  exhausts the pool with every sequence stuck, while reserving an answer
  budget at admission completes the same seven requests;
* invariants on random traces: pool accounting, row budget, FCFS, prefill
  before decode, contiguous positions, every request completing.
"""
import random

import pytest

from oracle import sched_sim as ss

SCALED = dict(block_size=4, max_slots=4, max_rows=12, chunk=8, answer_budget=16,
              max_blocks_per_seq=64)
PROMPTS = [3, 9, 14, 5, 8, 12, 6]
MAXTOK = [16, 12, 16, 8, 16, 10, 16]


def run(s, rng, check=None):
    steps = 0
    while s.running or s.waiting:
        p = s.plan()
        if check:
            check(s, p)
        s.commit([rng.randrange(50) for _ in p.sampled])
        steps += 1
        assert steps < 10000
    return steps


def test_hand_worked_plan():
    s = ss.Scheduler(ss.SchedConfig(n_blocks=16, **SCALED))
    A = ss.Request(0, [10, 11, 12, 13, 14, 15, 16, 17, 18, 19], 3)
    B = ss.Request(1, [20, 21, 22], 2)
    s.submit(A)
    s.submit(B)
    # step 1: both admitted (A slot 0, needs blocks(10+3)=4; B slot 1, needs 2).
    # A's first chunk = 8 prompt rows on blocks 0, 1; B's whole prompt (3 rows,
    # block 2) fits the remaining 4 rows and samples its last row.
    p = s.plan()
    assert p.resets == [0, 1]
    assert p.rows == [(0, 10 + i, i, 1, 0) for i in range(8)] + \
                     [(1, 20, 0, 1, 0), (1, 21, 1, 1, 0), (1, 22, 2, 1, 1)]
    assert p.sampled == [(1, 0)]
    assert p.block_tables == {0: [0, 1], 1: [2]}
    s.commit([77])
    # step 2: A's last 2 prompt rows (block 3 for positions 8-9, sample pos 9),
    # then B's decode row: token 77 at position 3 (still block 2).
    p = s.plan()
    assert p.rows == [(0, 18, 8, 1, 0), (0, 19, 9, 1, 1), (1, 77, 3, 0, 1)]
    assert p.sampled == [(0, 0), (1, 1)]
    assert p.block_tables == {0: [0, 1, 3], 1: [2]}
    assert s.commit([5, 6]) == [(1, ss.FINISH_LENGTH)]       # B has 2 tokens
    # step 3: A decodes token 5 at position 10; B's block 2 is free again.
    p = s.plan()
    assert p.rows == [(0, 5, 10, 0, 1)]
    assert p.sampled == [(0, 1)]
    assert sorted(s.free) == [2] + list(range(4, 16))
    assert s.finished[1] == (ss.FINISH_LENGTH, [77, 6])


def test_free_slot_admission_deadlocks_reservation_does_not():
    for reserve, expect_deadlock in ((False, True), (True, False)):
        s = ss.Scheduler(ss.SchedConfig(n_blocks=12, reserve_answer=reserve,
                                        stall_fallback=False, **SCALED))
        for i in range(7):
            s.submit(ss.Request(i, list(range(PROMPTS[i])), MAXTOK[i]))
        if expect_deadlock:
            with pytest.raises(ss.Deadlock):
                run(s, random.Random(1))
            st = s.stats()
            assert st["free_blocks"] == 0 and st["running"] == 4
        else:
            run(s, random.Random(1))
            assert all(s.finished[i] [0] == ss.FINISH_LENGTH and len(s.finished[i][1]) == MAXTOK[i]
                       for i in range(7))


def test_fallback_stops_youngest_when_budget_is_exceeded():
    """max_tokens beyond the answer budget can still exhaust the pool; the
    stall fallback then stops the youngest sequence (never the oldest)."""
    s = ss.Scheduler(ss.SchedConfig(n_blocks=12, **{**SCALED, "answer_budget": 4}))
    for i in range(4):
        s.submit(ss.Request(i, list(range(8)), 40))
    run(s, random.Random(2))
    reasons = {i: s.finished[i][0] for i in range(4)}
    assert ss.FINISH_LENGTH_FALLBACK in reasons.values()
    assert reasons[0] == ss.FINISH_LENGTH
    assert s.n_fallback >= 1


def make_checker(cfg, submitted_order):
    state = {"admitted": [], "next_pos": {}}

    def check(s, p):
        st = s.stats()
        assert st["allocated"] + st["outstanding"] <= cfg.n_blocks
        assert len(p.rows) <= cfg.max_rows
        kinds = [r[3] for r in p.rows]
        assert kinds == sorted(kinds, reverse=True)        # prefill rows first
        for r in s.running:
            if r.admit_seq >= len(state["admitted"]):
                state["admitted"].append(r.id)
        assert state["admitted"] == submitted_order[:len(state["admitted"])]   # FCFS
        by_slot = {}
        for slot, tok, pos, pre, smp in p.rows:
            by_slot.setdefault(slot, []).append(pos)
            assert pos < len(p.block_tables[slot]) * cfg.block_size
        req_of_slot = {r.slot: r for r in s.running}
        for slot, ps in by_slot.items():
            r = req_of_slot[slot]
            first = state["next_pos"].get(r.id, 0)
            assert ps == list(range(first, first + len(ps)))   # contiguous, continuing
            state["next_pos"][r.id] = first + len(ps)
        tables = [b for t in p.block_tables.values() for b in t]
        assert len(tables) == len(set(tables))               # no shared blocks
    return check


@pytest.mark.parametrize("seed", range(6))
def test_random_trace_invariants(seed):
    rng = random.Random(seed)
    cfg = ss.SchedConfig(n_blocks=rng.choice([40, 80, 400]), block_size=rng.choice([4, 32]),
                         max_slots=rng.choice([3, 8]), max_rows=rng.choice([16, 64]),
                         chunk=rng.choice([8, 32]), answer_budget=rng.choice([8, 64]),
                         max_blocks_per_seq=400)
    s = ss.Scheduler(cfg)
    order = []
    for i in range(40):
        P = rng.randint(1, 60)
        m = rng.randint(1, cfg.answer_budget)
        try:
            s.submit(ss.Request(i, [rng.randrange(100) for _ in range(P)], m))
            order.append(i)
        except ss.PoolTooSmall:
            pass
    run(s, rng, make_checker(cfg, order))
    assert sorted(s.finished) == sorted(order)
    assert all(v[0] == ss.FINISH_LENGTH for v in s.finished.values())
    assert s.stats()["free_blocks"] == cfg.n_blocks


def test_submit_rejects_requests_that_never_fit():
    s = ss.Scheduler(ss.SchedConfig(n_blocks=4, **SCALED))
    with pytest.raises(ss.PoolTooSmall):
        s.submit(ss.Request(0, list(range(15)), 16))      # blocks(15+16) = 8 > 4
    s.submit(ss.Request(1, list(range(3)), 5))           # blocks(8) = 2 fits
