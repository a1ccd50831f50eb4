"""GPU: the serving loop (C++ scheduler + engine) over a request trace.

Continuous batching must not change what any request generates: every
request's greedy tokens equal those of the oracle generating that request
alone (fp64, contiguous KV), outside near ties -- under the prefill-first
policy and under the Albatross policy, whose steps are composed differently
("大模型推理为什么需要 Continuous Batching", section 2.2: batching leaves each
sequence's output unchanged; "RWKV Runner Albatross 后端", worker main loop).
Also: a queue bound and a slow client on the GPU path end requests the way
the scheduler's rules say, and the blocks all come back.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import continuous_batching_decode_gb300 as cbd
    from continuous_batching_decode_gb300 import serve, synth
    from oracle import model as om
    from tests import gpu_util as gu

GREEDY = dict(temperature=0.0, top_p=1.0, top_k=0, frequency_penalty=0.0, presence_penalty=0.0,
              penalty_decay=1.0, seed=3)


@pytest.fixture(scope="module")
def tiny():
    from continuous_batching_decode_gb300 import build
    build.build()
    m = gu.Model("tiny", max_rows=64, max_slots=4, mbps=8)
    yield m
    m.close()


def trace(vocab, seed=0):
    rng = np.random.default_rng(seed)
    lens = [3, 9, 12, 40, 5, 20, 7, 33, 10, 64]
    return [dict(id=i, arrival=0.002 * i, prompt=synth.random_tokens(rng, P, vocab),
                 max_tokens=int(rng.integers(3, 9)), sampling=dict(GREEDY)) for i, P in enumerate(lens)]


def oracle_generate(model, prompt, n):
    """Greedy generation of one request alone; stops trusting the sequence at
    the first near tie (top-two gap < 1e-3)."""
    kv = {0: om.SequenceKV(model.cfg, len(prompt) + n + 1)}
    z = om.prefill(model, kv, 0, prompt)
    out = []
    for k in range(n):
        top = np.sort(z)[-2:]
        if top[1] - top[0] < 1e-3:
            return out, True
        t = int(np.argmax(z))
        out.append(t)
        if k + 1 < n:
            z = om.step(model, kv, [(0, t, len(prompt) + k, 1)])[0]
    return out, False


@pytest.mark.parametrize("policy", ["forma", "albatross"])
def test_trace_tokens_match_oracle_per_request(tiny, policy):
    reqs = trace(tiny.shape["vocab"])
    pool = tiny.pool(32)
    srv = serve.Server(tiny.e, pool.p, n_blocks=32, max_slots=4, max_rows=64, max_blocks_per_seq=8,
                       vocab=tiny.shape["vocab"], block_size=32, chunk=16, answer_budget=16, policy=policy)
    try:
        res = srv.run(reqs, step_ms=1.0)
    finally:
        srv.close()
        pool.close()
    assert all(res["outcome"][r["id"]] == cbd.FINISH_LENGTH for r in reqs)
    assert res["stats"]["free_blocks"] == 32
    model = tiny.oracle()
    compared = 0
    for r in reqs:
        want, tie = oracle_generate(model, r["prompt"], r["max_tokens"])
        got = res["tokens"][r["id"]]
        assert len(got) == r["max_tokens"]
        assert got[: len(want)] == want, f"request {r['id']}"
        compared += len(want)
    assert compared >= sum(r["max_tokens"] for r in reqs) - 4


def test_policies_generate_the_same_tokens(tiny):
    reqs = trace(tiny.shape["vocab"], seed=1)
    toks = {}
    for policy in ("forma", "albatross"):
        pool = tiny.pool(32)
        srv = serve.Server(tiny.e, pool.p, n_blocks=32, max_slots=4, max_rows=64, max_blocks_per_seq=8,
                           vocab=tiny.shape["vocab"], block_size=32, chunk=16, answer_budget=16, policy=policy)
        try:
            res = srv.run(reqs, step_ms=1.0)
        finally:
            srv.close()
            pool.close()
        toks[policy] = res["tokens"]
        assert res["steps"] > 0
    # the steps are composed differently, the ids are not (up to a near tie)
    model = tiny.oracle()
    for r in reqs:
        want, _ = oracle_generate(model, r["prompt"], r["max_tokens"])
        k = len(want)
        assert toks["forma"][r["id"]][:k] == toks["albatross"][r["id"]][:k] == want


def test_busy_and_slow_client_on_the_gpu_path(tiny):
    reqs = trace(tiny.shape["vocab"], seed=2)
    for r in reqs:
        r["arrival"] = 0.0
        r["max_tokens"] = 8
    pool = tiny.pool(32)
    srv = serve.Server(tiny.e, pool.p, n_blocks=32, max_slots=4, max_rows=64, max_blocks_per_seq=8,
                       vocab=tiny.shape["vocab"], block_size=32, chunk=16, answer_budget=16,
                       queue_per_slot=1, out_buffer=4)
    try:
        res = srv.run(reqs, step_ms=1.0)          # nobody reads: every admitted request lags out
    finally:
        srv.close()
        pool.close()
    oc = res["outcome"]
    assert sum(1 for v in oc.values() if v == "busy") == len(reqs) - 4    # 4 slots x 1 waiter
    admitted = [r["id"] for r in reqs if oc[r["id"]] != "busy"]
    assert all(oc[i] == cbd.FINISH_LAGGING for i in admitted)
    assert all(len(res["tokens"][i]) == 4 for i in admitted)
    assert res["stats"]["free_blocks"] == 32
