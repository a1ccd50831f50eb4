"""CPU tests of the C ABI: the library builds, loads and exports every
entry point include/cbd.h declares; host-only entry points (the scheduler)
match the Python policy simulator plan for plan; calls that need a GPU fail
with a status instead of crashing when there is none."""
import os
import random
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def cbd():
    from continuous_batching_decode_gb300 import build
    build.build()
    import continuous_batching_decode_gb300 as c
    c.lib()
    return c


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "cbd.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cbd_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(cbd):
    L = cbd.lib()
    names = declared_symbols()
    assert len(names) >= 20
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(cbd._cbd.PROTOS), "binding prototypes out of sync with the header"


def test_version_and_error_string(cbd):
    assert "sm_103a" in cbd.version()
    with pytest.raises(cbd.CbdError):
        cbd.sched_create(n_blocks=0)
    assert "out of range" in cbd.last_error()


def test_engine_create_without_gpu_fails_cleanly(cbd):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from continuous_batching_decode_gb300 import synth
    shape = synth.MODEL_SHAPES["tiny"]
    w = {k: v for k, v in synth.make_weights(shape, 0).items()}
    cfg = cbd.make_config(shape, 8, 4, 4)
    with pytest.raises(cbd.CbdError) as ei:
        cbd.engine_create(cfg, w)
    assert ei.value.status in (cbd.ECUDA, cbd.EUNSUPPORTED)


def test_config_validation_precedes_device(cbd):
    from continuous_batching_decode_gb300 import synth
    shape = dict(synth.MODEL_SHAPES["tiny"], head_dim=96)
    cfg = cbd.make_config(shape, 8, 4, 4)
    w = {k: v for k, v in synth.make_weights(synth.MODEL_SHAPES["tiny"], 0).items()}
    with pytest.raises(cbd.CbdError) as ei:
        cbd.engine_create(cfg, w)
    assert ei.value.status == cbd.EUNSUPPORTED


# ------------------------------------------------------------------ scheduler
def run_both(cbd, cfg_kw, reqs, seed, max_steps=5000):
    """Drive the C++ scheduler and the simulator with the same trace and the
    same fed-back tokens; assert identical plans at every step."""
    from oracle import sched_sim as ss
    sim = ss.Scheduler(ss.SchedConfig(**cfg_kw))
    h = cbd.sched_create(**cfg_kw)
    try:
        for rid, prompt, mt in reqs:
            err_c = err_s = None
            try:
                cbd.sched_submit(h, rid, prompt, mt, dict(temperature=1.0, top_p=0.3, seed=7, request_id=rid))
            except cbd.CbdError as e:
                err_c = e.status
            try:
                sim.submit(ss.Request(rid, list(prompt), mt))
            except ss.PoolTooSmall:
                err_s = cbd.EPOOL
            assert err_c == err_s
        rng = random.Random(seed)
        steps = 0
        W = cfg_kw["max_blocks_per_seq"]
        while sim.running or sim.waiting:
            p_s = sim.plan()
            p_c = cbd.sched_plan(h)
            assert p_c["rows"] == p_s.rows, f"step {steps}"
            assert p_c["sampled_ids"] == [i for i, _ in p_s.sampled]
            assert [s["token_index"] for s in p_c["sampling"]] == [t for _, t in p_s.sampled]
            assert all(s["request_id"] == i for s, i in zip(p_c["sampling"], p_c["sampled_ids"]))
            assert p_c["resets"] == p_s.resets
            assert p_c["stopped"] == [i for i, _ in p_s.stopped]
            for slot in range(cfg_kw["max_slots"]):
                want = p_s.block_tables.get(slot, [])
                assert p_c["n_blocks_per_slot"][slot] == len(want)
                assert list(p_c["block_tables"][slot][: len(want)]) == want
                assert all(p_c["block_tables"][slot][len(want):] == -1)
            toks = [rng.randrange(1000) for _ in p_s.sampled]
            fin_s = sim.commit(toks)
            fin_c = cbd.sched_commit(h, toks)
            assert [(i, r) for i, r, _ in fin_c] == fin_s
            st = cbd.sched_stats(h)
            ss_ = sim.stats()
            for k in ("running", "waiting", "free_blocks", "allocated", "reserved", "outstanding"):
                assert st[k] == ss_[k], k
            steps += 1
            assert steps < max_steps
        for rid, _, _ in reqs:
            if rid in sim.finished:
                assert cbd.sched_output(h, rid) == sim.finished[rid][1]
        return steps, sim
    finally:
        cbd.sched_destroy(h)


def trace(seed, n, vocab=1000, max_prompt=60, max_out=40):
    rng = random.Random(seed)
    return [(i, [rng.randrange(vocab) for _ in range(rng.randint(1, max_prompt))], rng.randint(1, max_out))
            for i in range(n)]


@pytest.mark.parametrize("policy", ["forma", "albatross"])
@pytest.mark.parametrize("seed", range(8))
def test_cpp_scheduler_matches_simulator(cbd, seed, policy):
    rng = random.Random(100 + seed)
    cfg = dict(n_blocks=rng.choice([12, 40, 200]), block_size=rng.choice([4, 32]), max_slots=rng.choice([3, 8, 16]),
               max_rows=rng.choice([12, 64]), chunk=rng.choice([8, 32]), answer_budget=rng.choice([8, 64]),
               max_blocks_per_seq=256, reserve_answer=True, stall_fallback=True, policy=policy)
    if policy == "albatross" and seed % 2:
        cfg.update(max_prefill=rng.choice([1, 3]), prefill_every=rng.choice([1, 3]), short_prompt=rng.choice([4, 20]))
    run_both(cbd, cfg, trace(seed, 30), seed)


def test_cpp_scheduler_fallback_path(cbd):
    cfg = dict(n_blocks=12, block_size=4, max_slots=4, max_rows=12, chunk=8, answer_budget=4,
               max_blocks_per_seq=64, reserve_answer=True, stall_fallback=True)
    reqs = [(i, list(range(8)), 40) for i in range(4)]
    _, sim = run_both(cbd, cfg, reqs, 3)
    assert sim.n_fallback >= 1


def test_cpp_scheduler_deadlock_on_free_slot_admission(cbd):
    """The page's scenario on its scaled constants: without the answer
    reservation the pool runs dry with every sequence stuck."""
    prompts = [3, 9, 14, 5, 8, 12, 6]
    maxt = [16, 12, 16, 8, 16, 10, 16]
    for reserve in (0, 1):
        h = cbd.sched_create(n_blocks=12, block_size=4, max_slots=4, max_rows=12, chunk=8, answer_budget=16,
                             max_blocks_per_seq=64, reserve_answer=reserve, stall_fallback=0)
        for i in range(7):
            cbd.sched_submit(h, i, list(range(prompts[i])), maxt[i])
        rng = random.Random(1)
        status = None
        for _ in range(500):
            try:
                p = cbd.sched_plan(h)
            except cbd.CbdError as e:
                status = e.status
                break
            if not p["rows"]:
                break
            cbd.sched_commit(h, [rng.randrange(50) for _ in p["sampling"]])
        st = cbd.sched_stats(h)
        cbd.sched_destroy(h)
        if reserve:
            assert status is None and st["running"] == 0 and st["waiting"] == 0
        else:
            assert status == cbd.EDEADLOCK and st["free_blocks"] == 0


def test_cpp_scheduler_rejects_bad_requests(cbd):
    h = cbd.sched_create(n_blocks=4, block_size=4, max_slots=2, max_rows=8, chunk=8, answer_budget=16,
                         max_blocks_per_seq=8)
    with pytest.raises(cbd.CbdError) as ei:
        cbd.sched_submit(h, 1, list(range(15)), 16)
    assert ei.value.status == cbd.EPOOL
    with pytest.raises(cbd.CbdError) as ei:
        cbd.sched_submit(h, 2, [], 4)
    assert ei.value.status == cbd.EINVAL
    cbd.sched_submit(h, 3, [1, 2], 3)
    with pytest.raises(cbd.CbdError) as ei:
        cbd.sched_submit(h, 3, [1, 2], 3)
    assert ei.value.status == cbd.EINVAL
    with pytest.raises(cbd.CbdError) as ei:
        cbd.sched_commit(h, [])
    assert ei.value.status == cbd.ESTATE
    cbd.sched_destroy(h)


@pytest.mark.parametrize("seed", range(6))
def test_cpp_scheduler_overload_matches_simulator(cbd, seed):
    """Bounded queue, wait budget, delivery buffers and aborts: the C++
    scheduler and the simulator, driven in lockstep by the same events
    (arrivals over a caller-driven clock, aborts between and during steps,
    clients that read or not), give the same plans and the same outcomes."""
    from oracle import sched_sim as ss
    rng = random.Random(500 + seed)
    kw = dict(n_blocks=rng.choice([40, 200]), block_size=4, max_slots=rng.choice([2, 6]),
              max_rows=rng.choice([16, 48]), chunk=8, answer_budget=16, max_blocks_per_seq=200,
              queue_per_slot=rng.choice([2, 8]), queue_timeout_ms=rng.choice([500, 3000]),
              out_buffer=rng.choice([2, 4]))
    sim = ss.Scheduler(ss.SchedConfig(**kw))
    h = cbd.sched_create(**kw)
    try:
        t, pending = 0, []
        for i in range(50):
            t += rng.choice([0, 10, 50])
            pending.append((t, i, [rng.randrange(100) for _ in range(rng.randint(1, 30))], rng.randint(1, 30)))
        slow = set(rng.sample(range(50), 5))
        t, steps = 0, 0
        while pending or sim.running or sim.waiting:
            t += rng.choice([5, 20, 200])
            sim.set_time(t)
            cbd.sched_set_time(h, t)
            while pending and pending[0][0] <= t:
                _, rid, prompt, mt = pending.pop(0)
                busy_s = busy_c = False
                try:
                    sim.submit(ss.Request(rid, prompt, mt))
                except ss.Busy:
                    busy_s = True
                try:
                    cbd.sched_submit(h, rid, prompt, mt)
                except cbd.CbdError as e:
                    assert e.status == cbd.EBUSY
                    busy_c = True
                assert busy_s == busy_c
            live = [r.id for r in sim.running] + [r.id for r in sim.waiting]
            if live and rng.random() < 0.05:
                victim = rng.choice(live)
                sim.abort(victim)
                cbd.sched_abort(h, victim)
            p_s = sim.plan()
            p_c = cbd.sched_plan(h)
            assert p_c["rows"] == p_s.rows, f"step {steps}"
            assert p_c["sampled_ids"] == [i for i, _ in p_s.sampled]
            assert p_c["resets"] == p_s.resets
            in_flight = [r.id for r in sim.running if not r.aborted]
            if in_flight and rng.random() < 0.05:
                victim = rng.choice(in_flight)
                sim.abort(victim)
                cbd.sched_abort(h, victim)
            toks = [rng.randrange(1000) for _ in p_s.sampled]
            fin_s = sim.commit(toks)
            fin_c = cbd.sched_commit(h, toks)
            assert [(i, r) for i, r, _ in fin_c] == fin_s
            assert cbd.sched_finished(h) == sim.take_finished()
            for r in list(sim.running):
                if r.id not in slow:
                    assert cbd.sched_read(h, r.id, 2) == sim.read(r.id, 2)
            st, ss_ = cbd.sched_stats(h), sim.stats()
            for k in ("running", "waiting", "free_blocks", "allocated", "reserved", "outstanding",
                      "rejected_busy", "timed_out", "aborted", "lagging"):
                assert st[k] == ss_[k], k
            steps += 1
            assert steps < 20000
        for rid in sim.finished:
            assert cbd.sched_output(h, rid) == sim.finished[rid][1]
            assert cbd.sched_read(h, rid) == sim.read(rid)
        with pytest.raises(cbd.CbdError):
            cbd.sched_set_time(h, t - 1)
    finally:
        cbd.sched_destroy(h)


def test_numpy_step_inputs_have_the_c_layout():
    """ROW_DTYPE / SAMPLING_DTYPE arrays are byte-for-byte the cbd_row /
    cbd_sampling arrays the C ABI reads, so step() may pass them as they are."""
    import ctypes
    import numpy as np
    from continuous_batching_decode_gb300 import _cbd as c
    assert c.ROW_DTYPE.itemsize == ctypes.sizeof(c.Row) == 20
    assert c.SAMPLING_DTYPE.itemsize == ctypes.sizeof(c.Sampling) == 48
    rows = [(1, 2, 3, 0, 1), (4, 5, 6, 1, 0), (7, 65535, 4095, 0, 1)]
    assert bytes(c.rows_table(rows).data) == bytes(c.rows_array(rows))
    sp = [dict(temperature=0.7, top_p=0.9, top_k=5, presence_penalty=0.1, frequency_penalty=0.2,
               penalty_decay=0.99, seed=2 ** 40 + 3, request_id=2 ** 33 + 7, token_index=9), dict()]
    assert bytes(c.sampling_table(sp).data) == bytes(c.sampling_array(sp))
    a, p, n = c._rows_arg(c.rows_table(rows))
    assert n == 3 and ctypes.addressof(p.contents) == a.ctypes.data
    with __import__("pytest").raises(TypeError):
        c._rows_arg(np.zeros(3, np.int32))
