"""GPU parity tests of the batched step through the C ABI (tiny decoder).

Oracle = the fp64 CPU decoder over contiguous KV.  Bars: logits max-abs
<= 1e-2 * max|z| and mean-abs <= 2e-3; greedy ids identical outside near
ties (top-two gap < 1e-3); sampled ids and counters bit-exact when the
oracle sampler runs on the GPU's own logits; paging and row order leave
every output bit-identical.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import continuous_batching_decode_gb300 as cbd
    from continuous_batching_decode_gb300 import synth
    from oracle import model as om
    from oracle import sampler as osamp
    from tests import gpu_util as gu


@pytest.fixture(scope="module", params=[(1, 1), (2, 0), (2, 2)],
                ids=["gemv+cuda_core_attn", "tcgen05+stream_attn", "tcgen05+chunk_attn"])
def tiny(request):
    """The tiny decoder with every contraction forced onto one GEMM path
    (1 = CUDA-core GEMV, 2 = tcgen05) and one attention kernel (1 = CUDA
    cores, 0 = persistent streaming mma.sync, 2 = one CTA per chunk)."""
    from continuous_batching_decode_gb300 import build
    build.build()
    m = gu.Model("tiny", max_rows=512, max_slots=8, mbps=16)
    cbd.engine_set_gemm_path(m.e, request.param[0])
    cbd.engine_set_attention_path(m.e, request.param[1])
    m.attn_path = request.param[1]
    yield m
    m.close()


def tiny_setup(tiny, placement_seed):
    """The tiny workload: slots 0-3 hold 5/17/33/64 prefilled positions;
    slot 4 gets a 40-token prompt chunk.  Returns pool, tables, rows, etc."""
    wl = synth.tiny_step(seed=0)
    need = {s: (c + 1 + 31) // 32 for s, c in enumerate(wl["contexts"])}
    need[4] = 2
    rng = np.random.default_rng(placement_seed)
    tables, nbps = synth.permuted_tables(need, wl["pool_blocks"], 16, rng)
    pool = tiny.pool(wl["pool_blocks"])
    for s, prior in enumerate(wl["prior"]):
        gu.gpu_prefill(tiny, pool, s, prior, tables, nbps, chunk=16)
    rows = [(s, wl["next_tokens"][s], c, 0, 1) for s, c in enumerate(wl["contexts"])]
    rows += [(4, t, i, 1, 1 if i == 39 else 0) for i, t in enumerate(wl["prompt"])]
    greedy = dict(temperature=0.0, penalty_decay=0.996, frequency_penalty=1.0, seed=1, request_id=10)
    sampled = dict(temperature=1.0, top_p=0.3, top_k=0, frequency_penalty=1.0, penalty_decay=0.996, seed=1234,
                   request_id=77, token_index=0)
    sampling = [dict(greedy, request_id=10 + s) for s in range(4)] + [sampled]
    return wl, pool, tables, nbps, rows, sampling


def preload_counters(tiny, wl):
    cv = gu.counters_view(tiny)
    cv.zero_()
    c = np.zeros(tiny.shape["vocab"], np.float32)
    for t in wl["replay"]:
        c = osamp.update_counters(c, t, 0.996)
    cv[4] = torch.from_numpy(c).cuda()
    return cv, c


def test_tiny_step_matches_oracle(tiny):
    wl, pool, tables, nbps, rows, sampling = tiny_setup(tiny, 1)
    cv, c4 = preload_counters(tiny, wl)
    pre = cv.cpu().numpy().copy()
    toks, z_gpu = gu.run_step(tiny, pool, rows, tables, nbps, sampling)
    post = cv.cpu().numpy()
    # oracle: prefill the same priors, then the same step
    om_ = tiny.oracle()
    kv = {s: om.SequenceKV(om_.cfg, 128) for s in range(5)}
    for s, prior in enumerate(wl["prior"]):
        om.prefill(om_, kv, s, prior)
    z = om.step(om_, kv, [(r[0], r[1], r[2], r[4]) for r in rows])
    mx, mean = gu.assert_logits_close(z_gpu, z, "tiny step")
    # greedy rows
    for j in range(4):
        if not gu.greedy_near_tie(z[j]):
            l2 = osamp.penalize(z_gpu[j].astype(np.float32), pre[j], 0.0, 1.0)
            assert toks[j] == int(np.argmax(l2))
            assert toks[j] == int(np.argmax(z[j]))
    # sampler on the GPU's own logits: bit-exact tokens and counters
    slots = [0, 1, 2, 3, 4]
    for j, s in enumerate(slots):
        p = gu.sampling_params(sampling[j])
        u = gu.uniform_of(sampling[j])
        lf = z_gpu[j].astype(np.float32)
        if not gu.sampling_near_tie(lf, pre[s], p, u):
            assert toks[j] == osamp.sample_row(lf, pre[s], p, u), f"row {j}"
        np.testing.assert_array_equal(post[s], osamp.update_counters(pre[s], int(toks[j]), p.penalty_decay))
    # KV written by the step and the prefill equals the oracle's bf16 KV.
    # Layer 0 depends only on the embedding and one GEMM: one bf16 ulp where
    # fp32 and fp64 round differently, plus a small absolute slack near zero
    # (the GEMM input carries ~2^-17 relative error from its hi/lo split).
    # Deeper layers inherit the layer-0 entries that rounded to different bf16
    # neighbours (each weighs ~1/context in attention), so they are bounded in
    # aggregate: a few ulps, and most entries identical.
    for s, c in enumerate(wl["contexts"] + [39]):
        n = c + 1
        K, V = pool.gather(tables, s, n)
        for l in range(om_.cfg.n_layers):
            for A, B in ((K[l], kv[s].K[l][:n]), (V[l], kv[s].V[l][:n])):
                rms = np.sqrt(np.mean(B * B))
                if l == 0:
                    tol = np.abs(B) * 2.0 ** -7 + 1e-4 * rms
                    assert np.mean(A != B) < 0.01, f"slot {s} layer 0: {np.mean(A != B):.3%} entries differ"
                else:
                    tol = np.abs(B) * 2.0 ** -5 + 2e-3 * rms
                    assert np.mean(A != B) < 0.15, f"slot {s} layer {l}: {np.mean(A != B):.3%} entries differ"
                bad = np.abs(A - B) > tol
                assert not bad.any(), f"slot {s} layer {l}: {bad.sum()} of {bad.size}, worst {np.abs(A - B).max():.3g}"
    # With the GPU's own KV as the oracle's prior state the only differences
    # left are the step's arithmetic: far inside the logit tolerance.
    prior = {s: c for s, c in enumerate(wl["contexts"])}
    kv2 = gu.oracle_kv_from_gpu(tiny, pool, tables, prior)
    kv2[4] = om.SequenceKV(om_.cfg, 64)
    z2 = om.step(om_, kv2, [(r[0], r[1], r[2], r[4]) for r in rows])
    err2 = np.abs(z_gpu - z2)
    assert err2.mean() <= 2e-4 and err2.max() <= 2e-3 * np.abs(z2).max(), (err2.mean(), err2.max())
    pool.close()
    print(f"tiny step: max-abs {mx:.3g} mean-abs {mean:.3g}; over GPU KV mean-abs {err2.mean():.3g}")


def test_paging_and_row_order_are_bit_exact(tiny):
    outs = []
    for placement in (1, 2):
        wl, pool, tables, nbps, rows, sampling = tiny_setup(tiny, placement)
        preload_counters(tiny, wl)
        toks, z = gu.run_step(tiny, pool, rows, tables, nbps, sampling)
        K0, V0 = pool.gather(tables, 3, 65)
        outs.append((toks, z, K0[1], V0[1]))
        if placement == 2:    # same placement, rows reversed
            preload_counters(tiny, wl)
            rr = rows[::-1]
            samp_r = [sampling[4]] + sampling[:4][::-1]
            pool2 = pool
            # rebuild the KV the reversed step overwrites with identical values
            toks_r, z_r = gu.run_step(tiny, pool2, rr, tables, nbps, samp_r)
            order = [4, 3, 2, 1, 0]
            np.testing.assert_array_equal(z_r[order], z)
            np.testing.assert_array_equal(toks_r[order], toks)
        pool.close()
    np.testing.assert_array_equal(outs[0][1], outs[1][1])
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][2], outs[1][2])
    np.testing.assert_array_equal(outs[0][3], outs[1][3])


def test_batched_equals_one_row_at_a_time(tiny):
    """Batching does not change results: the step's rows run one per step
    (prompt rows in order) give the same logits, bit for bit, with the
    prefill attention kernel off (the streaming kernel sums every row the
    same way whatever else is in the step); with it on (the default), the
    40-row prompt chunk is summed in blocks and the logits agree within the
    tolerance."""
    wl, pool, tables, nbps, rows, sampling = tiny_setup(tiny, 3)
    g = [dict(temperature=0.0)] * 5
    toks_on, z_on = gu.run_step(tiny, pool, rows, tables, nbps, g)
    pool.close()
    cbd.engine_set_prefill_attention(tiny.e, False)
    try:
        wl, pool, tables, nbps, rows, sampling = tiny_setup(tiny, 3)
        toks_b, z_b = gu.run_step(tiny, pool, rows, tables, nbps, g)
        pool.close()
        wl, pool, tables, nbps, rows, sampling = tiny_setup(tiny, 3)
        zs = []
        for r in rows:
            t, z = gu.run_step(tiny, pool, [r], tables, nbps, [dict(temperature=0.0)] if r[4] else [])
            if r[4]:
                zs.append(z[0])
        pool.close()
    finally:
        cbd.engine_set_prefill_attention(tiny.e, True)
    zs = np.array(zs)
    gu.assert_logits_close(zs, z_b, "batched vs single")
    np.testing.assert_array_equal(zs, z_b)
    gu.assert_logits_close(z_on, z_b, "prefill kernel on vs off")


def test_batched_equals_independent_sequences(tiny):
    """A batched step equals its sequences run as independent steps (each
    slot's rows alone: the 40-row prompt chunk as one step, each decode row
    as one), bit for bit, on the default path -- the prompt chunk takes the
    prefill attention kernel in both, and a row's result there does not
    depend on the other rows ("0.8MB 跑通 Qwen 第 14-1 篇", section 3:
    batching left the outputs byte-identical)."""
    wl, pool, tables, nbps, rows, sampling = tiny_setup(tiny, 4)
    g = [dict(temperature=0.0)] * 5
    toks_b, z_b = gu.run_step(tiny, pool, rows, tables, nbps, g)
    pool.close()
    wl, pool, tables, nbps, rows, sampling = tiny_setup(tiny, 4)
    zs, ts = [], []
    for slot in sorted({r[0] for r in rows}):
        part = [r for r in rows if r[0] == slot]
        m = sum(1 for r in part if r[4])
        t, z = gu.run_step(tiny, pool, part, tables, nbps, [dict(temperature=0.0)] * m)
        zs += list(z)
        ts += list(t)
    pool.close()
    np.testing.assert_array_equal(np.array(zs), z_b)
    np.testing.assert_array_equal(np.array(ts), toks_b)


def test_chunked_prefill_on_gpu(tiny):
    V = tiny.shape["vocab"]
    prompt = list(np.random.default_rng(5).integers(0, V, 40))
    tables = np.array([[3, 7] + [0] * 14], np.int32)
    nbps = np.array([2], np.int32)
    res = []
    for chunk in (40, 8, 1):
        pool = tiny.pool(8)
        gu.gpu_prefill(tiny, pool, 0, prompt[:-1], tables, nbps, chunk=chunk)
        _, z = gu.run_step(tiny, pool, [(0, prompt[-1], 39, 1, 1)], tables, nbps, [dict(temperature=0.0)])
        res.append(z[0])
        pool.close()
    for z in res[1:]:
        gu.assert_logits_close(z[None], res[0][None], "chunking")
    om_ = tiny.oracle()
    kv = {0: om.SequenceKV(om_.cfg, 64)}
    zo = om.prefill(om_, kv, 0, prompt, chunk=8)
    gu.assert_logits_close(res[0][None], zo[None], "chunked vs oracle")


def test_sampler_matches_oracle_on_gpu_logits(tiny):
    rng = np.random.default_rng(9)
    V = tiny.shape["vocab"]
    cv = gu.counters_view(tiny)
    configs = [dict(temperature=0.0, frequency_penalty=1.0, penalty_decay=0.996),
               dict(temperature=1.0, top_p=0.3, frequency_penalty=1.0, penalty_decay=0.996),
               dict(temperature=0.7, top_p=0.9, top_k=50, presence_penalty=0.5, frequency_penalty=0.3,
                    penalty_decay=0.99),
               dict(temperature=1.3, top_p=1.0, top_k=0),
               dict(temperature=1.0, top_k=1),
               dict(temperature=2.0, top_p=0.05, top_k=7)]
    mism = 0
    checked = 0
    for trial in range(12):
        m = 6
        lg = (rng.normal(0, 2.0, (m, V))).astype(np.float32)
        lg[:, :5] = lg[:, 5:10]                      # exact ties in value
        c0 = np.where(rng.random((8, V)) < 0.05, rng.integers(1, 5, (8, V)), 0).astype(np.float32)
        cv.copy_(torch.from_numpy(c0).cuda())
        slots = list(rng.permutation(8)[:m])
        samp = [dict(configs[j % len(configs)], seed=trial, request_id=1000 + j, token_index=trial) for j in range(m)]
        use_u = trial % 2 == 0
        us = [float(rng.random()) for _ in range(m)] if use_u else None
        out = torch.zeros(m, dtype=torch.int32, device="cuda")
        cbd.sample(tiny.e, torch.from_numpy(lg).cuda(), slots, samp, us, out)
        cbd.engine_check(tiny.e)
        toks = out.cpu().numpy()
        post = cv.cpu().numpy()
        for j in range(m):
            p = gu.sampling_params(samp[j])
            u = us[j] if use_u else gu.uniform_of(samp[j])
            s = slots[j]
            checked += 1
            if gu.sampling_near_tie(lg[j], c0[s], p, u):
                continue
            want = osamp.sample_row(lg[j], c0[s], p, u)
            mism += int(toks[j] != want)
            np.testing.assert_array_equal(post[s], osamp.update_counters(c0[s], int(toks[j]), p.penalty_decay))
    assert mism == 0, f"{mism} of {checked} sampled ids differ"


def test_philox_on_gpu_matches_host(tiny):
    """Draws with Philox on the device equal draws with the host Philox
    uniforms passed in (full distribution, so every bit of u matters)."""
    rng = np.random.default_rng(10)
    V = tiny.shape["vocab"]
    m = 8
    for trial in range(16):
        lg = torch.from_numpy(rng.normal(0, 0.5, (m, V)).astype(np.float32)).cuda()
        samp = [dict(temperature=1.0, top_p=1.0, seed=2 ** 40 + trial, request_id=2 ** 33 + j, token_index=trial * 3)
                for j in range(m)]
        us = [gu.uniform_of(s) for s in samp]
        a = torch.zeros(m, dtype=torch.int32, device="cuda")
        b = torch.zeros(m, dtype=torch.int32, device="cuda")
        cbd.sample(tiny.e, lg, list(range(m)), samp, None, a)
        cbd.sample(tiny.e, lg, list(range(m)), samp, us, b)
        np.testing.assert_array_equal(a.cpu().numpy(), b.cpu().numpy())


def test_step_validation(tiny):
    pool = tiny.pool(8)
    tok = torch.zeros(4, dtype=torch.int32, device="cuda")
    tables = np.array([[0, 1] + [0] * 14, [2, 3] + [0] * 14], np.int32)
    nbps = np.array([2, 2], np.int32)
    g = [dict(temperature=0.0)]
    ok = [(0, 1, 0, 1, 0), (0, 2, 1, 1, 1)]
    cbd.step(tiny.e, pool.p, ok, tables, nbps, g, None, tok)
    bad_cases = [
        ([(0, 1, 64, 0, 1)], tables, nbps, g),                    # pos beyond the slot's blocks
        ([(0, 99999, 0, 0, 1)], tables, nbps, g),                 # token out of range
        ([(0, 1, 0, 1, 0), (0, 1, 2, 1, 1)], tables, nbps, g),    # gap in positions
        ([(0, 1, 0, 1, 0), (0, 1, 0, 1, 1)], tables, nbps, g),    # repeated position
        ([(0, 1, 0, 1, 1), (0, 1, 1, 1, 1)], tables, nbps, g * 2),  # two sampled rows, one slot
        ([(0, 1, 0, 0, 1), (1, 1, 0, 0, 1)], np.array([[0, 1] + [0] * 14, [1, 3] + [0] * 14], np.int32), nbps, g * 2),
        ([(0, 1, 0, 0, 1)], np.array([[0, 9] + [0] * 14, [2, 3] + [0] * 14], np.int32), nbps, g),  # block outside pool
        ([(5, 1, 0, 0, 1)], tables, nbps, g),                     # slot outside the table
        ([(0, 1, 0, 0, 1)], tables, nbps, [dict(temperature=-1.0)]),
        ([(0, 1, 0, 0, 1)], tables, nbps, [dict(temperature=1.0, top_p=1.5)]),
    ]
    for rows, tb, nb, sp in bad_cases:
        with pytest.raises(cbd.CbdError) as ei:
            cbd.step(tiny.e, pool.p, rows, tb, nb, sp, None, tok)
        assert ei.value.status == cbd.EINVAL, rows
    cbd.engine_check(tiny.e)
    pool.close()


def test_gemm_paths_agree_on_long_prefill(tiny):
    """A 300-row prefill chunk (several 128-row N tiles on the tensor-core
    path) gives the oracle's logits on either GEMM path."""
    V = tiny.shape["vocab"]
    prompt = list(np.random.default_rng(21).integers(0, V, 300))
    tables = np.array([list(np.random.default_rng(22).permutation(16)[:10]) + [0] * 6], np.int32)
    nbps = np.array([10], np.int32)
    pool = tiny.pool(16)
    rows = [(0, t, i, 1, 1 if i == 299 else 0) for i, t in enumerate(prompt)]
    toks, z = gu.run_step(tiny, pool, rows, tables, nbps, [dict(temperature=0.0)])
    pool.close()
    om_ = tiny.oracle()
    kv = {0: om.SequenceKV(om_.cfg, 320)}
    zo = om.prefill(om_, kv, 0, prompt)
    gu.assert_logits_close(z, zo[None], "300-row prefill")


def test_multi_chunk_rows_and_l2_prefetch(tiny):
    """Rows whose context spans several 128-position attention chunks (so
    the chunk partials are merged) match the oracle; turning the L2
    prefetch off leaves every logit bit-identical (a prefetch is a cache
    hint only); a separate RMSNorm launch instead of the fused one agrees
    within the logit tolerance."""
    V = tiny.shape["vocab"]
    rng = np.random.default_rng(31)
    prompts = [list(rng.integers(0, V, 300)), list(rng.integers(0, V, 200))]
    perm = list(rng.permutation(16))
    tables = np.zeros((2, 16), np.int32)
    tables[0, :10] = perm[:10]
    tables[1, :6] = perm[10:16]
    tables[1, 6] = 16
    nbps = np.array([10, 7], np.int32)
    pool = tiny.pool(18)
    for s, p in enumerate(prompts):
        gu.gpu_prefill(tiny, pool, s, p[:-1], tables, nbps)
    rows = [(0, prompts[0][-1], 299, 0, 1), (1, prompts[1][-1], 199, 0, 1)]
    g = [dict(temperature=0.0)] * 2
    res = []
    for nbytes in (48 << 20, 0, 1 << 20):
        cbd.engine_set_l2_prefetch(tiny.e, nbytes)
        _, z = gu.run_step(tiny, pool, rows, tables, nbps, g)
        res.append(z)
    cbd.engine_set_l2_prefetch(tiny.e, 0)
    # RMSNorm folded into the GEMM epilogues vs a separate norm launch:
    # the same sums, rounded at different points
    cbd.engine_set_fused_norm(tiny.e, False)
    _, z_unfused = gu.run_step(tiny, pool, rows, tables, nbps, g)
    cbd.engine_set_fused_norm(tiny.e, True)
    pool.close()
    for z in res[1:]:
        np.testing.assert_array_equal(z, res[0])
    gu.assert_logits_close(z_unfused, res[0], "fused vs separate RMSNorm")
    om_ = tiny.oracle()
    zo = []
    for s, p in enumerate(prompts):
        kv = {s: om.SequenceKV(om_.cfg, 320)}
        zo.append(om.prefill(om_, kv, s, p))
    gu.assert_logits_close(res[0], np.array(zo), "multi-chunk rows")


def test_forbidden_tokens_on_gpu(tiny):
    """The engine's forbidden-token mask: ids the oracle sampler (step 0,
    forbidden ids removed before the penalty) gives for the same logits,
    counters and uniforms; forbidden ids never drawn; counters updated the
    same way; clearing the mask restores the unmasked draw."""
    rng = np.random.default_rng(21)
    V = tiny.shape["vocab"]
    cv = gu.counters_view(tiny)
    configs = [dict(temperature=0.0, frequency_penalty=1.0, penalty_decay=0.996),
               dict(temperature=1.0, top_p=0.3, frequency_penalty=1.0, penalty_decay=0.996),
               dict(temperature=0.8, top_p=0.95, top_k=20, presence_penalty=0.5, penalty_decay=0.99)]
    m = 6
    mism = checked = 0
    try:
        for trial in range(8):
            lg = rng.normal(0, 2.0, (m, V)).astype(np.float32)
            c0 = np.where(rng.random((8, V)) < 0.05, rng.integers(1, 5, (8, V)), 0).astype(np.float32)
            # forbid every row's top few raw logits plus random ids
            bad = sorted(set(np.argsort(-lg, axis=1)[:, :3].ravel().tolist()) |
                         set(rng.choice(V, 40, replace=False).tolist()))
            cbd.engine_set_forbidden(tiny.e, bad)
            cv.copy_(torch.from_numpy(c0).cuda())
            slots = list(rng.permutation(8)[:m])
            samp = [dict(configs[j % 3], seed=trial, request_id=500 + j, token_index=trial) for j in range(m)]
            us = [float(rng.random()) for _ in range(m)]
            out = torch.zeros(m, dtype=torch.int32, device="cuda")
            cbd.sample(tiny.e, torch.from_numpy(lg).cuda(), slots, samp, us, out)
            cbd.engine_check(tiny.e)
            toks = out.cpu().numpy()
            post = cv.cpu().numpy()
            assert not set(toks.tolist()) & set(bad)
            for j in range(m):
                p = gu.sampling_params(samp[j])
                s = slots[j]
                np.testing.assert_array_equal(post[s], osamp.update_counters(c0[s], int(toks[j]), p.penalty_decay))
                checked += 1
                if gu.sampling_near_tie(osamp.mask_forbidden(lg[j], bad), c0[s], p, us[j]):
                    continue
                mism += int(toks[j] != osamp.sample_row(lg[j], c0[s], p, us[j], forbidden=bad))
        assert mism == 0, f"{mism} of {checked} ids differ"
        # cleared: the greedy row takes its raw argmax again
        cbd.engine_set_forbidden(tiny.e, [])
        cv.zero_()
        lg = rng.normal(0, 2.0, (1, V)).astype(np.float32)
        out = torch.zeros(1, dtype=torch.int32, device="cuda")
        cbd.sample(tiny.e, torch.from_numpy(lg).cuda(), [0], [dict(temperature=0.0)], None, out)
        assert int(out.cpu()[0]) == int(np.argmax(lg[0]))
        with pytest.raises(cbd.CbdError):
            cbd.engine_set_forbidden(tiny.e, list(range(V)))       # nothing left to draw
        with pytest.raises(cbd.CbdError):
            cbd.engine_set_forbidden(tiny.e, [V])
    finally:
        cbd.engine_set_forbidden(tiny.e, [])


def oracle_over_gpu_kv(tiny, wl, pool, tables, rows):
    """The oracle's logits for the tiny step, with the GPU's prior KV as its
    state (the only differences left are the step's own arithmetic)."""
    om_ = tiny.oracle()
    prior = {s: c for s, c in enumerate(wl["contexts"])}
    kv = gu.oracle_kv_from_gpu(tiny, pool, tables, prior)
    kv[4] = om.SequenceKV(om_.cfg, 64)
    return om.step(om_, kv, [(r[0], r[1], r[2], r[4]) for r in rows])


def assert_tokens_match_oracle(tiny, toks, z_gpu, pre, sampling):
    """Sampled ids equal the oracle sampler's on the GPU's own logits
    (outside near ties)."""
    for j in range(len(toks)):
        p = gu.sampling_params(sampling[j])
        u = gu.uniform_of(sampling[j])
        lf = z_gpu[j].astype(np.float32)
        if not gu.sampling_near_tie(lf, pre[j], p, u):
            assert toks[j] == osamp.sample_row(lf, pre[j], p, u), f"row {j}"


def test_batch_graph_replay_is_bit_identical(tiny):
    """cbd_batch_set_graph: the captured graph replays the same kernels, so
    tokens and logits are bit-identical to the launch-by-launch run; a
    changed engine setting or output pointer captures a new graph.  The
    replayed step is also held to the oracle: logits within the tolerance,
    sampled ids equal to the oracle sampler's on the replayed logits."""
    wl, pool, tables, nbps, rows, sampling = tiny_setup(tiny, 3)
    cv = gu.counters_view(tiny)
    V = tiny.shape["vocab"]
    m = sum(1 for r in rows if r[4])
    b = cbd.batch_create(tiny.e, pool.p, rows, tables, nbps, sampling)
    try:
        def run(lg):
            cv.zero_()
            tok = torch.zeros(m, dtype=torch.int32, device="cuda")
            cbd.batch_run(tiny.e, pool.p, b, tok, lg)
            cbd.engine_check(tiny.e)
            return tok.cpu().numpy(), lg.cpu().numpy()
        lg1 = torch.zeros(m, V, dtype=torch.float32, device="cuda")
        t0, z0 = run(lg1)
        cbd.batch_set_graph(b, True)
        for _ in range(3):
            t, z = run(lg1)
            np.testing.assert_array_equal(t, t0)
            np.testing.assert_array_equal(z, z0)
        assert cbd.batch_captures(b) == 1
        zo = oracle_over_gpu_kv(tiny, wl, pool, tables, rows)
        gu.assert_logits_close(z.astype(np.float64), zo, "graph-replayed batch")
        assert_tokens_match_oracle(tiny, t, z.astype(np.float64), np.zeros((m, V), np.float32), sampling)
        cbd.engine_set_attention_path(tiny.e, tiny.attn_path)
        t, z = run(lg1)                      # a setting changed: captured again
        assert cbd.batch_captures(b) == 2
        np.testing.assert_array_equal(z, z0)
        lg2 = torch.zeros(m, V, dtype=torch.float32, device="cuda")
        t, z = run(lg2)                      # another output buffer: captured again
        assert cbd.batch_captures(b) == 3
        np.testing.assert_array_equal(t, t0)
        np.testing.assert_array_equal(z, z0)
        cbd.batch_set_graph(b, False)
        t, z = run(lg1)
        np.testing.assert_array_equal(z, z0)
    finally:
        cbd.batch_destroy(b)
        pool.close()


def test_step_graph_is_bit_identical(tiny):
    """cbd_engine_set_step_graph: cbd_step uploads and runs through cached
    graphs with results bit-identical to the launch-by-launch step; one
    capture per (shape, staging buffer), reused afterwards.  The graph-run
    step is also held to the oracle (logits and sampled ids)."""
    wl, pool, tables, nbps, rows, sampling = tiny_setup(tiny, 5)
    cv = gu.counters_view(tiny)
    V = tiny.shape["vocab"]
    m = sum(1 for r in rows if r[4])
    tok = torch.zeros(m, dtype=torch.int32, device="cuda")
    lg = torch.zeros(m, V, dtype=torch.float32, device="cuda")

    def run(rws):
        cv.zero_()
        k = sum(1 for r in rws if r[4])
        cbd.step(tiny.e, pool.p, rws, tables, nbps, sampling[:k], None, tok, lg)
        cbd.engine_check(tiny.e)
        return tok[:k].cpu().numpy(), lg[:k].cpu().numpy()
    try:
        t0, z0 = run(rows)
        c0 = cbd.engine_step_graph_captures(tiny.e)
        cbd.engine_set_step_graph(tiny.e, True)
        for i in range(4):
            t, z = run(rows)
            np.testing.assert_array_equal(t, t0)
            np.testing.assert_array_equal(z, z0)
        assert cbd.engine_step_graph_captures(tiny.e) - c0 == 2        # one per staging buffer
        zo = oracle_over_gpu_kv(tiny, wl, pool, tables, rows)
        gu.assert_logits_close(z.astype(np.float64), zo, "graph-run step")
        assert_tokens_match_oracle(tiny, t, z.astype(np.float64), np.zeros((m, V), np.float32), sampling)
        short = rows[:3]                                                # another shape: new graphs
        ts, zs = run(short)
        ts, zs = run(short)
        assert cbd.engine_step_graph_captures(tiny.e) - c0 == 4
        t, z = run(rows)                                                # the first shape is still cached
        assert cbd.engine_step_graph_captures(tiny.e) - c0 == 4
        np.testing.assert_array_equal(z, z0)
        cbd.engine_set_step_graph(tiny.e, False)
        t1, z1 = run(short)
        np.testing.assert_array_equal(z1, zs)
    finally:
        cbd.engine_set_step_graph(tiny.e, False)
        pool.close()
