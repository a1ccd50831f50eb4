"""GPU: the persistent contraction chain (cbd_engine_set_gemm_chain).

A decode step's O, gate/up and down contractions and the next layer's QKV
run as the phases of one launch.  Each phase keeps the per-launch kernel's
tiles, K split, reduction order and epilogue, so the step's results must be
bit-identical with the chain on and off -- the logits, the sampled ids, the
KV entries the step appends -- over several consecutive steps (the grid
barriers' counters are re-zeroed by each step's first kernel), on cbd_step
and on a resident batch replayed as a CUDA graph.  The per-launch path
itself is held to the oracle by the other parity tests; here the chain on
the full 7B shape is also checked against the oracle directly.  The
profile confirms which path ran: one gemm_chain launch per layer with the
chain on, none with it off."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import continuous_batching_decode_gb300 as cbd
    from continuous_batching_decode_gb300 import synth
    from oracle import model as om
    from tests import gpu_util as gu


def decode_setup(m, B, lo, hi, seed):
    s = m.shape
    db = synth.decode_batch(B, lo, hi, s["vocab"], seed)
    ctx = db["contexts"]
    need = {i: (c + 1 + 31) // 32 + 2 for i, c in enumerate(ctx)}      # room for a few steps
    n_pool = sum(need.values()) + 4
    tables, nbps = synth.permuted_tables(need, n_pool, m.mbps, np.random.default_rng(seed + 1))
    pool = m.pool(n_pool)
    gen = torch.Generator(device="cuda").manual_seed(seed + 3)
    for l in range(s["n_layers"]):
        v = torch.randn(pool.view[l].shape, generator=gen, device="cuda") * 1.3
        if pool.fp8:
            pool.view[l].copy_(v.to(torch.float8_e4m3fn).view(torch.uint8))
        else:
            pool.view[l].copy_(v.to(torch.bfloat16))
    return db, ctx, tables, nbps, pool


def run_steps(m, pool, db, ctx, tables, nbps, n_steps, chain, samp):
    """n_steps decode steps from the same starting state; per step the
    sampled ids and the logits, and the pool's bytes at the end."""
    cbd.engine_set_gemm_chain(m.e, chain)
    cv = gu.counters_view(m)
    cv.zero_()
    B = len(ctx)
    toks = np.asarray(db["tokens"][:B])
    out = []
    cbd.engine_profile(m.e, True)
    for k in range(n_steps):
        rows = [(i, int(toks[i]), ctx[i] + k, 0, 1) for i in range(B)]
        sp = [dict(s, token_index=k) for s in samp]
        t, z = gu.run_step(m, pool, rows, tables, nbps, sp)
        out.append((t, z))
        toks = t
    prof = cbd.engine_profile_read(m.e)
    cbd.engine_profile(m.e, False)
    return out, pool.view.clone(), prof


CASES = [
    # name, layers, rows, context range, kv_fp8
    ("tiny", None, 1, (3, 40), False),
    ("tiny", None, 7, (3, 200), False),
    ("tiny", None, 64, (1, 300), False),
    ("hd128", None, 33, (30, 500), False),
    ("hd128", None, 16, (30, 500), True),
    ("1b", 3, 32, (100, 1000), False),
    ("7b", 2, 1, (256, 4096), False),
    ("7b", 2, 32, (256, 4096), False),
]


@pytest.mark.parametrize("name,layers,B,ctx_range,fp8", CASES)
def test_chain_is_bit_identical_to_per_launch(name, layers, B, ctx_range, fp8):
    from continuous_batching_decode_gb300 import build
    build.build()
    hi = ctx_range[1]
    m = gu.Model(name, max_rows=64, max_slots=B, mbps=(hi + 4 + 31) // 32 + 2, layers=layers, kv_fp8=fp8)
    try:
        db, ctx, tables, nbps, pool = decode_setup(m, B, ctx_range[0], hi, seed=B)
        samp = [dict(temperature=0.8, top_p=0.9, top_k=0, frequency_penalty=0.5, penalty_decay=0.99, seed=5,
                     request_id=i) for i in range(B)]
        start = pool.view.clone()
        off, kv_off, prof_off = run_steps(m, pool, db, ctx, tables, nbps, 3, False, samp)
        pool.view.copy_(start)
        on, kv_on, prof_on = run_steps(m, pool, db, ctx, tables, nbps, 3, True, samp)
        L = m.shape["n_layers"]
        assert prof_off.get("gemm_chain", (0, 0))[0] == 0
        chained = prof_on.get("gemm_chain", (0, 0))[0]
        print(f"{name} B={B}: {chained} chain launches over 3 steps, per-launch GEMMs "
              f"{prof_on.get('gemm_o', (0, 0))[0]}")
        if name in ("tiny", "7b"):
            assert chained == 3 * L, prof_on
            assert prof_on.get("gemm_o", (0, 0))[0] == 0
            # layer 0's QKV once per step, plus the layers whose QKV K split
            # does not fit the chain's clusters
            assert 3 <= prof_on.get("gemm_qkv", (0, 0))[0] <= 3 * L
        for k, ((t0, z0), (t1, z1)) in enumerate(zip(off, on)):
            np.testing.assert_array_equal(z1, z0, err_msg=f"step {k} logits")
            np.testing.assert_array_equal(t1, t0, err_msg=f"step {k} ids")
        assert torch.equal(kv_on, kv_off), "KV pool after the steps"
        pool.close()
    finally:
        m.close()


def test_chain_graph_replay_matches_per_launch_step():
    """A resident batch replayed as a graph with the chain equals cbd_step
    without it, replay after replay."""
    from continuous_batching_decode_gb300 import build
    build.build()
    B = 24
    m = gu.Model("7b", max_rows=64, max_slots=B, mbps=(2048 + 31) // 32 + 2, layers=2)
    try:
        db, ctx, tables, nbps, pool = decode_setup(m, B, 100, 2000, seed=11)
        samp = [dict(temperature=0.0, seed=1, request_id=i) for i in range(B)]
        start = pool.view.clone()
        rows = [(i, int(db["tokens"][i]), ctx[i], 0, 1) for i in range(B)]
        cbd.engine_set_gemm_chain(m.e, False)
        t_ref, z_ref = gu.run_step(m, pool, rows, tables, nbps, samp)
        b = cbd.batch_create(m.e, pool.p, rows, tables, nbps, samp)
        try:
            tok_d = torch.zeros(B, dtype=torch.int32, device="cuda")
            lg_d = torch.zeros(B, m.shape["vocab"], dtype=torch.float32, device="cuda")
            pool.view.copy_(start)
            cbd.batch_run(m.e, pool.p, b, tok_d, lg_d)
            cbd.engine_check(m.e)
            launches_off = cbd.batch_launches(b)
            cbd.engine_set_gemm_chain(m.e, True)
            cbd.batch_set_graph(b, True)
            for it in range(3):
                pool.view.copy_(start)
                cbd.batch_run(m.e, pool.p, b, tok_d, lg_d)
                cbd.engine_check(m.e)
                np.testing.assert_array_equal(lg_d.cpu().numpy().astype(np.float64), z_ref, err_msg=f"replay {it}")
                np.testing.assert_array_equal(tok_d.cpu().numpy(), t_ref)
            assert cbd.batch_captures(b) == 1
            # per layer O, gate/up and down become one chain (which may also
            # take the next layer's QKV)
            L = m.shape["n_layers"]
            assert 2 * L <= launches_off - cbd.batch_launches(b) <= 3 * L - 1
        finally:
            cbd.batch_destroy(b)
        pool.close()
    finally:
        m.close()


def test_chain_7b_all_layers_against_oracle():
    """The full 32-layer 7B shape with the chain switched on against the
    oracle on 8 of 32 decode rows: logits within the tolerance."""
    from continuous_batching_decode_gb300 import build
    build.build()
    B = 32
    m = gu.Model("7b", max_rows=B, max_slots=B, mbps=(4096 + 1 + 31) // 32 + 2)
    try:
        db, ctx, tables, nbps, pool = decode_setup(m, B, 256, 4096, seed=0)
        cbd.engine_set_gemm_chain(m.e, True)
        rows = [(i, int(db["tokens"][i]), ctx[i], 0, 1) for i in range(B)]
        samp = [dict(temperature=0.0, seed=0, request_id=i) for i in range(B)]
        cbd.engine_profile(m.e, True)
        _, z = gu.run_step(m, pool, rows, tables, nbps, samp)
        prof = cbd.engine_profile_read(m.e)
        cbd.engine_profile(m.e, False)
        assert prof.get("gemm_chain", (0, 0))[0] == m.shape["n_layers"], prof
        grp = [0, 5, 9, 14, 18, 23, 27, 31]
        kv = gu.oracle_kv_from_gpu(m, pool, tables, {i: ctx[i] for i in grp})
        zr = om.step(m.oracle(cache=False), kv, [(i, rows[i][1], ctx[i], 1) for i in grp])
        mx, mean = gu.assert_logits_close(z[grp], zr, "7B chain")
        print(f"7B chain vs oracle, 8 rows: max-abs {mx:.3g} mean-abs {mean:.3g}")
        pool.close()
    finally:
        m.close()
