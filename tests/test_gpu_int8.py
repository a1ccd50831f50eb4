"""GPU parity with int8 weights (cbd_config.weights_int8; "RWKV Runner
Albatross 后端", 边界与后续路线 lists int8-quantised weights as follow-up work).

The reading (per output row, symmetric: s = fp32(max|w| / 127), q = nearest
integer to w / s, ties to even, clamped to +-127; embedding and gains
unchanged) is the oracle's quantize_int8_rows, pinned on the CPU.  Here:
  * the engine's int8 matrices and scales, read back through
    cbd_engine_read_weight, equal the oracle's quantisation bit for bit
    (integer work: the bar is exact), in the engine's row order;
  * the step's logits meet the tolerance (max-abs <= 1e-2 * max|z|,
    mean-abs <= 2e-3) against the oracle run over q * s -- tiny (own KV and
    GPU KV), 1B (32 decode rows) and the 7B shape at two layers (32 decode
    rows over contexts U[256, 4096]) -- and sampled ids and counters equal
    the oracle sampler's on the GPU's logits, outside near ties."""
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
    from tests.test_gpu_step import tiny_setup


def engine_rows(shape, which, w, l):
    """A streamed matrix of the synthetic weights in the engine's row order
    (bf16 bit arrays -> fp64)."""
    b = lambda k: om.bf16_bits_to_f64(synth.bf16_bits(w[k]))
    hd, hq, hkv = shape["head_dim"], shape["n_heads"], shape["n_kv_heads"]
    if which == cbd.WEIGHT_QKV:
        m = np.concatenate([b(f"{l}.wq"), b(f"{l}.wk"), b(f"{l}.wv")])
        perm = np.arange(m.shape[0])
        half = hd // 2
        for h in range(hq + hkv):
            for i in range(half):
                perm[h * hd + 2 * i] = h * hd + i
                perm[h * hd + 2 * i + 1] = h * hd + i + half
        return m[perm]
    if which == cbd.WEIGHT_O:
        return b(f"{l}.wo")
    if which == cbd.WEIGHT_GATE_UP:
        g, u = b(f"{l}.w_gate"), b(f"{l}.w_up")
        m = np.empty((2 * g.shape[0], g.shape[1]))
        m[0::2], m[1::2] = g, u
        return m
    if which == cbd.WEIGHT_DOWN:
        return b(f"{l}.w_down")
    return b("lm_head")


@pytest.mark.parametrize("name", ["tiny", "1b"])
def test_int8_weights_equal_oracle_quantisation(name):
    from continuous_batching_decode_gb300 import build
    build.build()
    m = gu.Model(name, max_rows=64, max_slots=8, mbps=8, weights_int8=True)
    try:
        layers = [0, m.shape["n_layers"] - 1]
        for which in (cbd.WEIGHT_QKV, cbd.WEIGHT_O, cbd.WEIGHT_GATE_UP, cbd.WEIGHT_DOWN, cbd.WEIGHT_LM_HEAD):
            for l in (layers if which != cbd.WEIGHT_LM_HEAD else [0]):
                ref = engine_rows(m.shape, which, m.w, l)
                q, s = om.quantize_int8_rows(ref)
                gq, gs = cbd.engine_read_weight(m.e, which, l, ref.shape[0], ref.shape[1], int8=True)
                np.testing.assert_array_equal(gs, s, err_msg=f"scales of matrix {which} layer {l}")
                np.testing.assert_array_equal(gq, q, err_msg=f"int8 matrix {which} layer {l}")
    finally:
        m.close()


def test_bf16_engine_weights_read_back_exactly():
    """The repacked bf16 arena is a faithful copy in the documented row order."""
    from continuous_batching_decode_gb300 import build
    build.build()
    m = gu.Model("tiny", max_rows=64, max_slots=8, mbps=8)
    try:
        for which in (cbd.WEIGHT_QKV, cbd.WEIGHT_O, cbd.WEIGHT_GATE_UP, cbd.WEIGHT_DOWN, cbd.WEIGHT_LM_HEAD):
            ref = engine_rows(m.shape, which, m.w, 1 if which != cbd.WEIGHT_LM_HEAD else 0)
            gb, _ = cbd.engine_read_weight(m.e, which, 1, ref.shape[0], ref.shape[1], int8=False)
            np.testing.assert_array_equal(om.bf16_bits_to_f64(gb), ref)
    finally:
        m.close()


def check_sampling(toks, z_gpu, post, pre, samp, rows_of=None):
    checked = 0
    for j in range(len(toks)):
        p = gu.sampling_params(samp[j])
        u = gu.uniform_of(samp[j])
        lf = z_gpu[j].astype(np.float32)
        if not gu.sampling_near_tie(lf, pre[j], p, u):
            assert toks[j] == osamp.sample_row(lf, pre[j], p, u), f"row {j}"
            checked += 1
        np.testing.assert_array_equal(post[j], osamp.update_counters(pre[j], int(toks[j]), p.penalty_decay))
    return checked


def test_int8_tiny_step_matches_oracle():
    from continuous_batching_decode_gb300 import build
    build.build()
    m = gu.Model("tiny", max_rows=512, max_slots=8, mbps=16, weights_int8=True)
    try:
        wl, pool, tables, nbps, rows, sampling = tiny_setup(m, 2)
        cv = gu.counters_view(m)
        cv.zero_()
        toks, z_gpu = gu.run_step(m, pool, rows, tables, nbps, sampling)
        post = cv.cpu().numpy()
        om_ = m.oracle()
        # oracle with its own KV (priors prefilled in fp64 over q * s)
        kv = {s: om.SequenceKV(om_.cfg, 128) for s in range(5)}
        for s, prior in enumerate(wl["prior"]):
            om.prefill(om_, kv, s, prior)
        z = om.step(om_, kv, [(r[0], r[1], r[2], r[4]) for r in rows])
        mx, mean = gu.assert_logits_close(z_gpu, z, "int8 tiny step")
        # and over the GPU's KV: only the step's own arithmetic differs
        prior = {s: c for s, c in enumerate(wl["contexts"])}
        kv2 = gu.oracle_kv_from_gpu(m, pool, tables, prior)
        kv2[4] = om.SequenceKV(om_.cfg, 64)
        z2 = om.step(om_, kv2, [(r[0], r[1], r[2], r[4]) for r in rows])
        err2 = np.abs(z_gpu - z2)
        assert err2.mean() <= 2e-4 and err2.max() <= 2e-3 * np.abs(z2).max(), (err2.mean(), err2.max())
        slots = [r[0] for r in rows if r[4]]
        check_sampling(toks, z_gpu, post[slots], np.zeros_like(post[slots]), sampling)
        pool.close()
        print(f"int8 tiny step: max-abs {mx:.3g} mean-abs {mean:.3g}; over GPU KV {err2.mean():.3g}")
    finally:
        m.close()


@pytest.mark.parametrize("name,layers,lo,hi", [("1b", None, 64, 2048), ("7b", 2, 256, 4096)],
                         ids=["1b", "7b_two_layers"])
def test_int8_decode_step_matches_oracle(name, layers, lo, hi):
    from continuous_batching_decode_gb300 import build
    build.build()
    B = 32
    mbps = (hi + 1 + 31) // 32
    m = gu.Model(name, max_rows=B, max_slots=B, mbps=mbps, layers=layers, weights_int8=True)
    try:
        s = m.shape
        db = synth.decode_batch(B, lo, hi, s["vocab"], seed=7)
        ctx = db["contexts"]
        need = {i: (c + 1 + 31) // 32 for i, c in enumerate(ctx)}
        n_pool = sum(need.values()) + 4
        tables, nbps = synth.permuted_tables(need, n_pool, mbps, np.random.default_rng(8))
        pool = m.pool(n_pool)
        gen = torch.Generator(device="cuda").manual_seed(9)
        for l in range(s["n_layers"]):
            pool.view[l].copy_((torch.randn(pool.view[l].shape, generator=gen, device="cuda") * 1.3)
                               .to(torch.bfloat16))
        cv = gu.counters_view(m)
        cv.zero_()
        rows = [(i, db["tokens"][i], ctx[i], 0, 1) for i in range(B)]
        samp = [dict(temperature=1.0, top_p=0.3, top_k=0, frequency_penalty=1.0, penalty_decay=0.996, seed=12,
                     request_id=700 + i, token_index=3) for i in range(B)]
        toks, z_gpu = gu.run_step(m, pool, rows, tables, nbps, samp)
        post = cv.cpu().numpy()
        om_ = m.oracle(cache=(name != "7b" or layers is not None))
        z = np.zeros((B, s["vocab"]))
        for g0 in range(0, B, 8):
            grp = list(range(g0, g0 + 8))
            kv = gu.oracle_kv_from_gpu(m, pool, tables, {i: ctx[i] for i in grp})
            z[grp] = om.step(om_, kv, [(rows[i][0], rows[i][1], rows[i][2], 1) for i in grp])
            del kv
        pool.close()
        mx, mean = gu.assert_logits_close(z_gpu, z, f"int8 {name} step")
        checked = check_sampling(toks, z_gpu, post[:B], np.zeros_like(post[:B]), samp)
        assert checked >= B - 2
        print(f"int8 {name} step: max-abs {mx:.3g} mean-abs {mean:.3g}")
    finally:
        m.close()
