"""Pins for the Albatross composition policy of the scheduler simulator
(page "RWKV Runner Albatross 后端", section 连续批处理：Worker 主循环), CPU only:

* at most max_prefill_count = max(int(batch * 0.125), 1) requests prefill at
  once (the page's formula, evaluated for several batch sizes);
* a prompt shorter than min_forward_seq_len = 10 is fed one token per step,
  a prompt of 10 or more by sequence chunks;
* sequence chunks come once after every decode_prefill_ratio = 5 steps that
  carry other rows, and at once when nothing else runs;
* invariants on random traces, and the same requests finishing with the
  same lengths under both policies.
"""
import random

import pytest

from oracle import sched_sim as ss

BASE = dict(block_size=4, max_rows=64, chunk=8, answer_budget=16, max_blocks_per_seq=128)


def cfg(**kw):
    d = dict(n_blocks=400, max_slots=16, policy="albatross")
    d.update(BASE)
    d.update(kw)
    return ss.SchedConfig(**d)


@pytest.mark.parametrize("slots,expect", [(4, 1), (7, 1), (8, 1), (16, 2), (31, 3), (32, 4), (64, 8)])
def test_max_prefill_count_formula(slots, expect):
    s = ss.Scheduler(cfg(max_slots=slots, n_blocks=4000))
    assert s.max_prefill == expect
    for i in range(slots):
        s.submit(ss.Request(i, list(range(40)), 3))          # long prompts: 5 chunks each
    p = s.plan()
    assert len(s.running) == expect                            # admission stops at the cap
    assert len({r[0] for r in p.rows}) == expect


def test_short_prompts_take_one_token_per_step():
    s = ss.Scheduler(cfg())
    s.submit(ss.Request(0, list(range(9)), 2))                 # 9 < 10: one-token prefill
    s.submit(ss.Request(1, list(range(10)), 2))                # 10: sequence prefill
    p = s.plan()
    assert [(r[0], r[2]) for r in p.rows if r[0] == 0] == [(0, 0)]
    assert [r[2] for r in p.rows if r[0] == 1] == list(range(8))   # one chunk of 8
    steps = 1
    while s.finished.get(0) is None:
        s.commit([5] * len(p.sampled))
        p = s.plan()
        steps += 1
        rows0 = [r for r in p.rows if r[0] == 0]
        assert len(rows0) <= 1
    assert steps >= 10                                         # 9 prompt steps + 1 decode step


def test_sequence_steps_are_paced_by_decode_rounds():
    s = ss.Scheduler(cfg(max_prefill=4))
    s.submit(ss.Request(0, [1, 2, 3], 60))                     # decodes throughout
    while not s.running or not s.running[0].generated:
        p = s.plan()
        s.commit([9] * len(p.sampled))
    s.submit(ss.Request(1, list(range(24)), 2))                # three chunks of 8
    seq_steps = []
    for step in range(40):
        p = s.plan()
        if any(r[0] != s.running[0].slot and r[3] == 1 for r in p.rows):
            seq_steps.append(step)
        s.commit([9] * len(p.sampled))
        if 1 in s.finished:
            break
    assert seq_steps == [0, 6, 12]                             # then 5 decode-only steps each time


def test_without_decode_rows_sequence_steps_run_back_to_back():
    s = ss.Scheduler(cfg())
    s.submit(ss.Request(0, list(range(24)), 1))
    chunks = []
    while 0 not in s.finished:
        p = s.plan()
        chunks.append(len(p.rows))
        s.commit([1] * len(p.sampled))
    assert chunks == [8, 8, 8]


@pytest.mark.parametrize("seed", range(5))
def test_random_traces_both_policies(seed):
    rng = random.Random(seed)
    kw = dict(n_blocks=rng.choice([60, 400]), max_slots=rng.choice([4, 16]), max_rows=rng.choice([16, 64]))
    reqs = [(i, [rng.randrange(100) for _ in range(rng.choice([3, 9, 12, 40]))], rng.randint(1, 20))
            for i in range(40)]
    lengths = {}
    for policy in ("forma", "albatross"):
        s = ss.Scheduler(cfg(policy=policy, **kw))
        for rid, prompt, mt in reqs:
            s.submit(ss.Request(rid, list(prompt), mt))
        trng = random.Random(seed)
        steps = 0
        while s.running or s.waiting:
            p = s.plan()
            kinds = [r[3] for r in p.rows]
            assert kinds == sorted(kinds, reverse=True)       # prefill rows first
            if policy == "albatross":
                pre = {r.id for r in s.running if r.n_prefilled < len(r.prompt)}
                assert len(pre) <= s.max_prefill
            st = s.stats()
            assert st["allocated"] + st["outstanding"] <= s.cfg.n_blocks
            s.commit([trng.randrange(100) for _ in p.sampled])
            steps += 1
            assert steps < 5000
        assert len(s.free) == s.cfg.n_blocks
        lengths[policy] = {rid: len(v[1]) for rid, v in s.finished.items()}
    assert lengths["forma"] == lengths["albatross"] == {rid: mt for rid, _, mt in reqs}
