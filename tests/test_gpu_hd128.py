"""GPU parity at head_dim 128 with 4 query heads per KV head -- the 7B
shape's attention instantiation -- on a 2-layer toy model, for bf16 and for
FP8 (E4M3) KV: logits against the fp64 oracle (prefilled from scratch, and
over the GPU's own KV), greedy ids outside near ties."""
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


@pytest.mark.parametrize("kv_fp8", [False, True], ids=["bf16_kv", "e4m3_kv"])
def test_hd128_decode_and_prefill_match_oracle(kv_fp8):
    from continuous_batching_decode_gb300 import build
    build.build()
    m = gu.Model("hd128", max_rows=256, max_slots=8, mbps=12, kv_fp8=kv_fp8)
    try:
        V = m.shape["vocab"]
        rng = np.random.default_rng(11)
        ctx = [5, 40, 100, 200, 31, 64, 129]
        need = {s: (c + 1 + 31) // 32 for s, c in enumerate(ctx)}
        need[7] = 2                                        # a 50-token prompt chunk in the step
        tables, nbps = synth.permuted_tables(need, 48, 12, rng)
        pool = m.pool(48)
        priors = [synth.random_tokens(rng, c, V) for c in ctx]
        for s, pr in enumerate(priors):
            gu.gpu_prefill(m, pool, s, pr, tables, nbps, chunk=64)
        toks = synth.random_tokens(rng, len(ctx), V)
        prompt = synth.random_tokens(rng, 50, V)
        rows = [(s, toks[s], c, 0, 1) for s, c in enumerate(ctx)]
        rows += [(7, t, i, 1, 1 if i == 49 else 0) for i, t in enumerate(prompt)]
        samp = [dict(GREEDY, request_id=s) for s in range(len(ctx) + 1)]
        got, z_gpu = gu.run_step(m, pool, rows, tables, nbps, samp)
        om_ = m.oracle()
        kv = {s: om.SequenceKV(om_.cfg, 256) for s in range(8)}
        for s, pr in enumerate(priors):
            om.prefill(om_, kv, s, pr)
        z = om.step(om_, kv, [(r[0], r[1], r[2], r[4]) for r in rows])
        gu.assert_logits_close(z_gpu, z, f"hd128 step ({'e4m3' if kv_fp8 else 'bf16'} KV)")
        for j in range(len(z)):
            if not gu.greedy_near_tie(z[j]):
                assert got[j] == int(np.argmax(z[j])), f"row {j}"
        kv2 = gu.oracle_kv_from_gpu(m, pool, tables, {s: c for s, c in enumerate(ctx)})
        kv2[7] = om.SequenceKV(om_.cfg, 64)
        z2 = om.step(om_, kv2, [(r[0], r[1], r[2], r[4]) for r in rows])
        err2 = np.abs(z_gpu - z2)
        assert err2.mean() <= 2e-4 and err2.max() <= 2e-3 * np.abs(z2).max(), (err2.mean(), err2.max())
        pool.close()
    finally:
        m.close()
