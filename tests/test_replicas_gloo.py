"""The multi-GPU mode (independent replicas) on CPU: two gloo ranks each run
the C++ scheduler on their round-robin share of one request trace, with
synthetic sampled tokens, and the host-side reductions combine them.  Checks
that every request is owned and finished exactly once, that each rank's
admission invariants hold, and the max / sum aggregation of bench.py."""
import os
import random

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from continuous_batching_decode_gb300 import replicas

WORLD = 2


def _trace(n=40, seed=7):
    rng = random.Random(seed)
    return [(i, [rng.randrange(1000) for _ in range(rng.choice([5, 20, 70]))], rng.randint(1, 30)) for i in range(n)]


def _rank_main(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import continuous_batching_decode_gb300 as cbd
        reqs = _trace()
        mine = replicas.route([r[0] for r in reqs], rank, WORLD)
        s = cbd.sched_create(n_blocks=48, block_size=32, max_slots=6, max_rows=96, chunk=32, answer_budget=16,
                             max_blocks_per_seq=16)
        by_id = {r[0]: r for r in reqs}
        for rid in mine:
            _, prompt, max_tokens = by_id[rid]
            cbd.sched_submit(s, rid, prompt, max_tokens)
        finished, steps, rows = {}, 0, 0
        while len(finished) < len(mine):
            p = cbd.sched_plan(s)
            steps += 1
            rows += len(p["rows"])
            assert steps < 10000, "replica did not drain"
            toks = [(rid * 31 + steps) % 1000 for rid in p["sampled_ids"]]
            for fid, reason, n_tok in cbd.sched_commit(s, toks):
                finished[fid] = n_tok
        st = cbd.sched_stats(s)
        cbd.sched_destroy(s)
        total_rows = replicas.sum_over_ranks(rows, dist)
        slowest = replicas.max_over_ranks(float(steps), dist)
        tput = replicas.job_throughput(float(rows), float(steps), dist)
        gathered = [None] * WORLD
        dist.all_gather_object(gathered, sorted(finished.items()))
        if rank == 0:
            out.put(dict(finished=gathered, total_rows=total_rows, slowest=slowest, tput=tput, stats=st))
        else:
            out.put(dict(rows=rows, steps=steps))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_drain_one_trace():
    pytest.importorskip("torch.distributed")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + random.Random(os.getpid()).randrange(2000)
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(WORLD)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    r0 = next(r for r in res if "finished" in r)
    r1 = next(r for r in res if "rows" in r)
    reqs = _trace()
    owners = {}
    for rank, fin in enumerate(r0["finished"]):
        for rid, n_tok in fin:
            assert rid not in owners, f"request {rid} finished on two ranks"
            owners[rid] = rank
            assert rid % WORLD == rank                      # round-robin ownership
            assert n_tok == reqs[rid][2]                    # ran to its max_tokens
    assert sorted(owners) == [r[0] for r in reqs]
    assert r0["slowest"] >= r1["steps"]
    assert r0["total_rows"] >= r1["rows"]
    assert r0["tput"] == pytest.approx(r0["total_rows"] / r0["slowest"])


def test_route_partitions_requests():
    ids = list(range(11))
    parts = [replicas.route(ids, r, 3) for r in range(3)]
    assert sorted(sum(parts, [])) == ids
    assert parts[1] == [1, 4, 7, 10]
    with pytest.raises(ValueError):
        replicas.route(ids, 3, 3)
