"""GPU parity of the 128-row-tile tensor-core GEMM (the kernel that steps of
many rows -- prefill chunks mixed with decode rows, "20.3 服务、批处理与流式"
section 20.3.2 -- run their weight contractions on).

It computes the same sums as the 64-row-tile kernel (fp32 accumulation of
bf16 weights times the hi + lo bf16 halves of the activations) in another
order, so: logits meet the oracle's tolerance with it forced on and off,
ragged last tiles included; two runs are bit-identical (no split-K, no
atomics); the K/V it appends equal the other kernel's up to one bf16 ulp.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import continuous_batching_decode_gb300 as cbd
    from continuous_batching_decode_gb300 import synth
    from oracle import model as om
    from tests import gpu_util as gu

GREEDY = dict(temperature=0.0, top_p=1.0, top_k=0, frequency_penalty=0.0, presence_penalty=0.0, penalty_decay=1.0)


@pytest.fixture(scope="module")
def tiny_tc():
    from continuous_batching_decode_gb300 import build
    build.build()
    m = gu.Model("tiny", max_rows=512, max_slots=8, mbps=16)
    cbd.engine_set_gemm_path(m.e, 2)
    yield m
    m.close()


def mixed_step(m, n_prompt, seed):
    """Slots 0-3 decode over 5/40/97/130 prefilled positions; slot 4 brings
    an n_prompt-token prompt chunk.  Returns (pool, tables, nbps, rows,
    sampling, priors, prompt)."""
    V = m.shape["vocab"]
    rng = np.random.default_rng(seed)
    ctx = [5, 40, 97, 130]
    need = {s: (c + 1 + 31) // 32 for s, c in enumerate(ctx)}
    need[4] = (n_prompt + 31) // 32
    n_pool = sum(need.values()) + 2
    tables, nbps = synth.permuted_tables(need, n_pool, 16, rng)
    pool = m.pool(n_pool)
    priors = [synth.random_tokens(rng, c, V) for c in ctx]
    for s, pr in enumerate(priors):
        gu.gpu_prefill(m, pool, s, pr, tables, nbps, chunk=64)
    toks = synth.random_tokens(rng, 4, V)
    prompt = synth.random_tokens(rng, n_prompt, V)
    rows = [(s, toks[s], c, 0, 1) for s, c in enumerate(ctx)]
    rows += [(4, t, i, 1, 1 if i == n_prompt - 1 else 0) for i, t in enumerate(prompt)]
    samp = [dict(GREEDY, request_id=s) for s in range(5)]
    return pool, tables, nbps, rows, samp, priors, prompt, ctx


@pytest.mark.parametrize("n_prompt", [41, 300], ids=["one_ragged_tile", "three_tiles"])
def test_rows_gemm_matches_oracle(tiny_tc, n_prompt):
    m = tiny_tc
    res = {}
    # the RMSNorm as its own kernel on both (the 128-row-tile kernel never
    # fuses it), so the two differ only in the order of the fp32 sums
    cbd.engine_set_fused_norm(m.e, False)
    for rows_min in (0, 1):                 # 0: 64-row-tile kernel; 1: 128-row-tile kernel
        cbd.engine_set_rows_gemm(m.e, rows_min, force=True)
        pool, tables, nbps, rows, samp, priors, prompt, ctx = mixed_step(m, n_prompt, 7)
        got, z = gu.run_step(m, pool, rows, tables, nbps, samp)
        K, V = pool.gather(tables, 4, n_prompt)
        res[rows_min] = (got, z, K[0], V[0])
        pool.close()
    cbd.engine_set_rows_gemm(m.e, 512, force=False)
    cbd.engine_set_fused_norm(m.e, True)
    om_ = m.oracle()
    kv = {s: om.SequenceKV(om_.cfg, 512) for s in range(5)}
    for s, pr in enumerate(priors):
        om.prefill(om_, kv, s, pr)
    zo = om.step(om_, kv, [(r[0], r[1], r[2], r[4]) for r in rows])
    for rows_min, (got, z, K, V) in res.items():
        gu.assert_logits_close(z, zo, f"{len(rows)}-row step, rows kernel {'on' if rows_min else 'off'}")
        for j in range(len(zo)):
            if not gu.greedy_near_tie(zo[j]):
                assert got[j] == int(np.argmax(zo[j])), f"row {j}"
    # layer 0's appended K/V of the prompt (same inputs on both kernels):
    # equal up to the order of the fp32 sums -- one bf16 ulp where the two
    # sums round to different sides, plus an allowance of 2^-14 * max|value|
    # for sums whose terms cancel (the fp32 error of a 256-term sum is up to
    # 256 * 2^-24 times the sum of the terms' magnitudes)
    for A, B in ((res[0][2], res[1][2]), (res[0][3], res[1][3])):
        ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(A), 1e-30))[1] - 8)
        tol = ulp * 1.0001 + 2.0 ** -14 * np.abs(A).max()
        bad = np.abs(A - B) > tol
        assert not bad.any(), (int(bad.sum()), float(np.abs(A - B).max()), float(np.abs(A).max()))
        assert np.mean(A != B) < 0.05, np.mean(A != B)


def test_rows_gemm_is_deterministic(tiny_tc):
    m = tiny_tc
    cbd.engine_set_rows_gemm(m.e, 1, force=True)
    outs = []
    for _ in range(2):
        pool, tables, nbps, rows, samp, *_ = mixed_step(m, 300, 9)
        got, z = gu.run_step(m, pool, rows, tables, nbps, samp)
        K, V = pool.gather(tables, 4, 300)
        outs.append((got, z, K, V))
        pool.close()
    cbd.engine_set_rows_gemm(m.e, 512, force=False)
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)


def test_rows_gemm_setting_is_validated(tiny_tc):
    with pytest.raises(cbd.CbdError):
        cbd.engine_set_rows_gemm(tiny_tc.e, -1)
    cbd.engine_set_rows_gemm(tiny_tc.e, 512)


@pytest.mark.parametrize("kv_fp8", [False, True], ids=["bf16_kv", "e4m3_kv"])
def test_rows_gemm_hd128(kv_fp8):
    """Head dim 128, 4 q heads per KV head (the 7B attention shape) with a
    200-row prompt chunk: the QKV epilogue's RoPE and K/V stores (bf16 or
    E4M3) from the 128-row-tile kernel against the oracle."""
    from continuous_batching_decode_gb300 import build
    build.build()
    m = gu.Model("hd128", max_rows=256, max_slots=8, mbps=12, kv_fp8=kv_fp8)
    try:
        cbd.engine_set_gemm_path(m.e, 2)
        cbd.engine_set_rows_gemm(m.e, 1, force=True)
        V = m.shape["vocab"]
        rng = np.random.default_rng(13)
        ctx = [5, 70, 150]
        need = {s: (c + 1 + 31) // 32 for s, c in enumerate(ctx)}
        need[3] = 7
        tables, nbps = synth.permuted_tables(need, 24, 12, rng)
        pool = m.pool(24)
        priors = [synth.random_tokens(rng, c, V) for c in ctx]
        for s, pr in enumerate(priors):
            gu.gpu_prefill(m, pool, s, pr, tables, nbps, chunk=64)
        toks = synth.random_tokens(rng, len(ctx), V)
        prompt = synth.random_tokens(rng, 200, V)
        rows = [(s, toks[s], c, 0, 1) for s, c in enumerate(ctx)]
        rows += [(3, t, i, 1, 1 if i == 199 else 0) for i, t in enumerate(prompt)]
        samp = [dict(GREEDY, request_id=s) for s in range(4)]
        got, z_gpu = gu.run_step(m, pool, rows, tables, nbps, samp)
        om_ = m.oracle()
        kv = {s: om.SequenceKV(om_.cfg, 256) for s in range(4)}
        for s, pr in enumerate(priors):
            om.prefill(om_, kv, s, pr)
        z = om.step(om_, kv, [(r[0], r[1], r[2], r[4]) for r in rows])
        gu.assert_logits_close(z_gpu, z, f"hd128 rows-kernel step ({'e4m3' if kv_fp8 else 'bf16'} KV)")
        for j in range(len(z)):
            if not gu.greedy_near_tie(z[j]):
                assert got[j] == int(np.argmax(z[j])), f"row {j}"
        pool.close()
    finally:
        m.close()


def test_rows_gemm_7b_shape_two_layers():
    """The 7B layer shapes (d 4096, 32 q / 8 KV heads of 128, ffn 14336;
    two layers) with a 512-row prompt chunk and 32 decode rows: logits of
    the sampled rows against the oracle with the 128-row-tile kernel where
    it fills the GPU (the default), on every GEMM (forced), and off."""
    from continuous_batching_decode_gb300 import build
    build.build()
    m = gu.Model("7b", max_rows=544, max_slots=33, mbps=17, layers=2)
    try:
        cbd.engine_set_gemm_path(m.e, 2)
        V = m.shape["vocab"]
        rng = np.random.default_rng(17)
        ctx = [int(c) for c in rng.integers(1, 64, 32)]
        need = {s: (c + 1 + 31) // 32 for s, c in enumerate(ctx)}
        need[32] = 16
        n_pool = sum(need.values()) + 2
        tables, nbps = synth.permuted_tables(need, n_pool, 17, rng)
        priors = [synth.random_tokens(rng, c, V) for c in ctx]
        toks = synth.random_tokens(rng, 32, V)
        prompt = synth.random_tokens(rng, 512, V)
        rows = [(s, toks[s], c, 0, 1) for s, c in enumerate(ctx)]
        rows += [(32, t, i, 1, 1 if i == 511 else 0) for i, t in enumerate(prompt)]
        samp = [dict(GREEDY, request_id=s) for s in range(33)]
        res = {}
        for name, (rows_min, force) in {"auto": (512, False), "forced": (1, True), "off": (0, False)}.items():
            cbd.engine_set_rows_gemm(m.e, rows_min, force=force)
            pool = m.pool(n_pool)
            for s, pr in enumerate(priors):
                gu.gpu_prefill(m, pool, s, pr, tables, nbps, chunk=64)
            res[name] = gu.run_step(m, pool, rows, tables, nbps, samp)
            pool.close()
        cbd.engine_set_rows_gemm(m.e, 512)
        om_ = m.oracle(cache=False)
        kv = {s: om.SequenceKV(om_.cfg, 544) for s in range(33)}
        for s, pr in enumerate(priors):
            om.prefill(om_, kv, s, pr)
        z = om.step(om_, kv, [(r[0], r[1], r[2], r[4]) for r in rows])
        for name, (got, zg) in res.items():
            gu.assert_logits_close(zg, z, f"7B-shape 2-layer 544-row step, rows kernel {name}")
            for j in range(len(z)):
                if not gu.greedy_near_tie(z[j]):
                    assert got[j] == int(np.argmax(z[j])), f"{name}: row {j}"
    finally:
        m.close()
