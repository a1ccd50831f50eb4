"""GPU parity over long contexts (the long-context decode configuration:
contexts up to 32768 positions, split across 128-position chunks and merged).

At the 7B shape the oracle cannot hold a 32K-position row's KV for 32
layers, so this runs the 7B shape's attention instantiation (head dim 128,
4 query heads per KV head) on the two-layer `hd128` model, at the full
context lengths: decode rows over 32767, 20000, 4096 and 5 cached positions
(256, 157, 32 and 1 chunks), the pool filled with seeded random K/V, bf16
and E4M3.  The oracle takes the GPU's KV as its state; logits must meet the
tolerance and greedy ids match outside near ties."""
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
def test_long_context_decode_matches_oracle(kv_fp8):
    from continuous_batching_decode_gb300 import build
    build.build()
    ctx = [32767, 20000, 4096, 5]
    mbps = (max(ctx) + 1 + 31) // 32
    m = gu.Model("hd128", max_rows=8, max_slots=4, mbps=mbps, kv_fp8=kv_fp8)
    try:
        V = m.shape["vocab"]
        rng = np.random.default_rng(23)
        need = {s: (c + 1 + 31) // 32 for s, c in enumerate(ctx)}
        n_pool = sum(need.values()) + 4
        tables, nbps = synth.permuted_tables(need, n_pool, mbps, rng)
        pool = m.pool(n_pool)
        gen = torch.Generator(device="cuda").manual_seed(29)
        for l in range(m.shape["n_layers"]):
            r = torch.randn(pool.view[l].shape, generator=gen, device="cuda") * 1.3
            pool.view[l].copy_(r.to(torch.float8_e4m3fn).view(torch.uint8) if kv_fp8 else r.to(torch.bfloat16))
        toks = synth.random_tokens(rng, len(ctx), V)
        rows = [(s, toks[s], c, 0, 1) for s, c in enumerate(ctx)]
        samp = [dict(GREEDY, request_id=s) for s in range(len(ctx))]
        got, z_gpu = gu.run_step(m, pool, rows, tables, nbps, samp)
        kv = gu.oracle_kv_from_gpu(m, pool, tables, {s: c for s, c in enumerate(ctx)})
        pool.close()
        z = om.step(m.oracle(), kv, [(r[0], r[1], r[2], r[4]) for r in rows])
        mx, mean = gu.assert_logits_close(z_gpu, z, f"long contexts ({'e4m3' if kv_fp8 else 'bf16'} KV)")
        print(f"long contexts {ctx}: max-abs {mx:.3g} mean-abs {mean:.3g}")
        for j in range(len(z)):
            if not gu.greedy_near_tie(z[j]):
                assert got[j] == int(np.argmax(z[j])), f"row {j}"
    finally:
        m.close()
