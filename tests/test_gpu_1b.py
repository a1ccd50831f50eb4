"""GPU parity at the 1B shape: 32 decode slots, contexts ~ U[64, 2048],
sampling T=1, top_p 0.3, frequency penalty 1, decay 0.996.

The prior KV is built on the GPU by prefilling random prompts through the
step itself (512-row chunks); the oracle then takes that KV (read back from
the paged pool into contiguous per-sequence arrays) as its initial state and
runs the same decode step in fp64.  Logits must meet the tolerance; sampled
ids and counters must match the oracle sampler run on the GPU's logits."""
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


@pytest.fixture(scope="module")
def m1b():
    from continuous_batching_decode_gb300 import build
    build.build()
    m = gu.Model("1b", max_rows=512, max_slots=32, mbps=65)
    yield m
    m.close()


def test_1b_decode_step(m1b):
    B = 32
    s = m1b.shape
    db = synth.decode_batch(B, 64, 2048, s["vocab"], seed=4)
    ctx = db["contexts"]
    need = {i: (c + 1 + 31) // 32 for i, c in enumerate(ctx)}
    n_pool = sum(need.values()) + 4
    tables, nbps = synth.permuted_tables(need, n_pool, 65, np.random.default_rng(5))
    pool = m1b.pool(n_pool)
    rng = np.random.default_rng(6)
    for i, c in enumerate(ctx):
        gu.gpu_prefill(m1b, pool, i, list(rng.integers(0, s["vocab"], c)), tables, nbps, chunk=512)
    cv = gu.counters_view(m1b)
    cv.zero_()
    pre = np.zeros((B, s["vocab"]), np.float32)
    for i in range(B):                       # replay 64 earlier tokens as generated
        c = pre[i]
        for t in rng.integers(0, s["vocab"], 64):
            c = osamp.update_counters(c, int(t), 0.996)
        pre[i] = c
    cv.copy_(torch.from_numpy(pre).cuda())
    rows = [(i, db["tokens"][i], ctx[i], 0, 1) for i in range(B)]
    samp = [dict(temperature=1.0, top_p=0.3, top_k=0, frequency_penalty=1.0, penalty_decay=0.996, seed=11,
                 request_id=500 + i, token_index=64) for i in range(B)]
    toks, z_gpu = gu.run_step(m1b, pool, rows, tables, nbps, samp)
    post = cv.cpu().numpy()
    kv = gu.oracle_kv_from_gpu(m1b, pool, tables, {i: c for i, c in enumerate(ctx)})
    pool.close()
    om_ = m1b.oracle(cache=False)
    z = om.step(om_, kv, [(r[0], r[1], r[2], 1) for r in rows])
    mx, mean = gu.assert_logits_close(z_gpu, z, "1B step")
    checked = 0
    for j in range(B):
        p = gu.sampling_params(samp[j])
        u = gu.uniform_of(samp[j])
        lf = z_gpu[j].astype(np.float32)
        if not gu.sampling_near_tie(lf, pre[j], p, u):
            assert toks[j] == osamp.sample_row(lf, pre[j], p, u), f"row {j}"
            checked += 1
        np.testing.assert_array_equal(post[j], osamp.update_counters(pre[j], int(toks[j]), 0.996))
    assert checked >= B - 2
    print(f"1B step: max-abs {mx:.3g} mean-abs {mean:.3g}")
