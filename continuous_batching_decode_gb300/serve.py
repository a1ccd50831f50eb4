"""Host serving loop: the C++ scheduler drives the engine over a request trace.

Every iteration ("20.3 服务、批处理与流式", section 20.3.2; "大模型推理为什么需要
Continuous Batching", sections 2.2 and 3.3): requests that have arrived are
submitted, the scheduler admits and composes the next step (prefill chunks and
one row per decoding sequence), newly admitted slots get their penalty
counters zeroed, the engine runs the step, and the sampled tokens are committed
back, which retires finished requests and frees their slots and blocks for the
next iteration.  All of the step's work runs in libcbd (CUDA kernels and the
C++ scheduler); this module only moves host arrays between the two and keeps
the clock.

The clock is the wall clock by default.  ``step_ms`` replaces it with a virtual
one that advances by a fixed amount per iteration (arrivals and queue timeouts
then replay exactly, e.g. in tests).
"""
from __future__ import annotations

import time

import numpy as np
import torch

from . import _cbd as C


class Server:
    """One engine, one KV pool and one scheduler.

    ``sched_kw`` are cbd_sched_config fields (see ``sched_create``); n_blocks,
    max_slots, max_rows and max_blocks_per_seq default to the engine's.
    """

    def __init__(self, engine, pool, n_blocks: int, max_slots: int, max_rows: int, max_blocks_per_seq: int,
                 vocab: int, **sched_kw):
        self.e, self.pool = engine, pool
        kw = dict(n_blocks=n_blocks, max_slots=max_slots, max_rows=max_rows, max_blocks_per_seq=max_blocks_per_seq)
        kw.update(sched_kw)
        self.sched = C.sched_create(**kw)
        self.max_slots = max_slots
        self.vocab = vocab
        self.out_tokens = torch.zeros(max(max_slots, 1) + max_rows, dtype=torch.int32, device="cuda")

    def close(self) -> None:
        if self.sched is not None:
            C.sched_destroy(self.sched)
            self.sched = None

    def run(self, requests, step_ms: float | None = None, max_steps: int = 10_000_000) -> dict:
        """Serve ``requests`` (dicts with id, arrival [s], prompt, max_tokens
        and optionally sampling) to completion.  Returns the generated tokens
        per request, each request's outcome, time to first token and finish
        time, and totals."""
        reqs = sorted(requests, key=lambda r: (r["arrival"], r["id"]))
        first_tok, done_at, outcome, arrival = {}, {}, {}, {}
        n_gen = 0
        steps = rows_total = 0
        t_sched = 0.0                      # host time in plan + commit (C++ scheduler + marshalling)
        t_start = time.perf_counter()
        vt = 0.0

        def now_s() -> float:
            return vt if step_ms is not None else time.perf_counter() - t_start

        i = 0
        running = 0
        while i < len(reqs) or running:
            t = now_s()
            C.sched_set_time(self.sched, int(t * 1000))
            while i < len(reqs) and reqs[i]["arrival"] <= t:
                r = reqs[i]
                i += 1
                arrival[r["id"]] = r["arrival"]
                samp = dict(r.get("sampling") or {})
                samp.setdefault("request_id", r["id"])
                try:
                    C.sched_submit(self.sched, r["id"], r["prompt"], r["max_tokens"], samp)
                except C.CbdError as ex:
                    if ex.status != C.EBUSY:
                        raise
                    outcome[r["id"]] = "busy"
            ts = time.perf_counter()
            p = C.sched_plan_raw(self.sched)       # the plan's arrays go to cbd_step as they are
            sampled = [p.sampled_ids[j] for j in range(p.n_sampled)]
            t_sched += time.perf_counter() - ts
            for j in range(p.n_resets):
                C.slot_reset(self.e, p.reset_slots[j])
            m = len(sampled)
            if p.n_rows:
                C.step_plan(self.e, self.pool, p, self.out_tokens)
                toks = self.out_tokens[:m].cpu().numpy().tolist() if m else []
                steps += 1
                rows_total += p.n_rows
            else:
                toks = []
                if i < len(reqs) and step_ms is None:        # idle until the next arrival
                    time.sleep(max(0.0, min(reqs[i]["arrival"] - now_s(), 0.01)))
            ts = time.perf_counter()
            fin = C.sched_commit(self.sched, toks)
            t_sched += time.perf_counter() - ts
            if step_ms is not None:
                vt += step_ms / 1000.0
            t = now_s()
            for rid in sampled:
                if rid not in first_tok:
                    first_tok[rid] = t
            n_gen += m
            for rid, why, _ in fin + C.sched_finished(self.sched):
                outcome[rid] = why
                done_at[rid] = t
            st = C.sched_stats(self.sched)
            running = st["running"] + st["waiting"]
            if steps > max_steps:
                raise RuntimeError("trace did not drain")
        wall = now_s()
        C.engine_check(self.e)
        out = {rid: C.sched_output(self.sched, rid) for rid, why in outcome.items() if why != "busy"}
        ttft = np.array([first_tok[r] - arrival[r] for r in first_tok if r in arrival])
        return dict(tokens=out, outcome=outcome, ttft=ttft, finish={r: done_at[r] - arrival[r] for r in done_at},
                    generated=n_gen, steps=steps, rows=rows_total, wall_s=wall,
                    sched_us_per_step=1e6 * t_sched / max(steps, 1),
                    tok_s=n_gen / wall if wall > 0 else float("nan"), stats=C.sched_stats(self.sched))
