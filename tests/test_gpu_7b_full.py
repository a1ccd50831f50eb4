"""GPU parity at the full 7B decode workload, in the bench's configuration:
32 layers (d 4096, 32 q / 8 KV heads of 128, ffn 14336, vocab 65536), 32
decode slots with contexts U[256, 4096] (seed 0), the KV pool filled with
random bf16 values, sampling T 1, top_p 0.3, frequency penalty 1, decay 0.996.

The oracle cannot run all 32 rows through 32 layers in seconds, so it takes
three of them -- the shortest, a median and the longest context -- with the
GPU's KV (read back from the paged pool) as their state, and computes their
logits one by one in fp64.  Logits must meet the tolerance; the sampled ids
must match the oracle sampler run on the GPU's logits (outside near ties) and
the counters its update."""
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


def test_7b_decode_step_sampled_rows():
    from continuous_batching_decode_gb300 import build
    build.build()
    B, lo, hi, seed = 32, 256, 4096, 0
    m = gu.Model("7b", max_rows=B, max_slots=B, mbps=(hi + 1 + 31) // 32)
    try:
        s = m.shape
        db = synth.decode_batch(B, lo, hi, s["vocab"], seed)
        ctx = db["contexts"]
        need = {i: (c + 1 + 31) // 32 for i, c in enumerate(ctx)}
        n_pool = sum(need.values()) + 8
        tables, nbps = synth.permuted_tables(need, n_pool, m.mbps, np.random.default_rng(seed + 1))
        pool = m.pool(n_pool)
        gen = torch.Generator(device="cuda").manual_seed(seed + 3)
        for l in range(s["n_layers"]):
            pool.view[l].copy_((torch.randn(pool.view[l].shape, generator=gen, device="cuda") * 1.3)
                               .to(torch.bfloat16))
        cv = gu.counters_view(m)
        cv.zero_()
        rows = [(i, db["tokens"][i], ctx[i], 0, 1) for i in range(B)]
        samp = [dict(temperature=1.0, top_p=0.3, top_k=0, frequency_penalty=1.0, penalty_decay=0.996, seed=seed,
                     request_id=i, token_index=0) for i in range(B)]
        toks, z_gpu = gu.run_step(m, pool, rows, tables, nbps, samp)
        post = cv.cpu().numpy()
        order = np.argsort(ctx)
        pick = [int(order[0]), int(order[B // 2]), int(order[-1])]
        kv = gu.oracle_kv_from_gpu(m, pool, tables, {i: ctx[i] for i in pick})
        pool.close()
        om_ = m.oracle(cache=False)
        z = om.step(om_, kv, [(rows[i][0], rows[i][1], rows[i][2], 1) for i in pick])
        mx, mean = gu.assert_logits_close(z_gpu[pick], z, "7B step (sampled rows)")
        print(f"7B step, rows {pick} (contexts {[ctx[i] for i in pick]}): max-abs {mx:.3g} mean-abs {mean:.3g}")
        pre = np.zeros(s["vocab"], np.float32)
        for i in pick:
            p = gu.sampling_params(samp[i])
            u = gu.uniform_of(samp[i])
            lf = z_gpu[i].astype(np.float32)
            if not gu.sampling_near_tie(lf, pre, p, u):
                assert toks[i] == osamp.sample_row(lf, pre, p, u), f"row {i}"
            np.testing.assert_array_equal(post[i], osamp.update_counters(pre, int(toks[i]), 0.996))
    finally:
        m.close()
