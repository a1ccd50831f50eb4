"""GPU parity at the full 7B decode workload, in the bench's configuration:
32 layers (d 4096, 32 q / 8 KV heads of 128, ffn 14336, vocab 65536), 32
decode slots with contexts U[256, 4096] (seed 0), the KV pool filled with
random bf16 values, sampling T 1, top_p 0.3, frequency penalty 1, decay 0.996.

The step runs twice, on the two paths a caller has: cbd_step (host arrays
staged and launched kernel by kernel), and the path the benchmark times --
a resident cbd_batch replayed as one CUDA graph (captured on the first run,
replayed on the second).  Batching must not change a row's result ("0.8MB
跑通 Qwen 第 14-1 篇", section 3: batched and serial runs gave the same
outputs), so the oracle computes every one of the 32 rows in fp64 with the
GPU's KV (read back from the paged pool) as its state.  For all 32 rows and
both paths the logits must meet the tolerance (max-abs <= 1e-2 * max|z|,
mean-abs <= 2e-3), the sampled ids must equal the oracle sampler's on the
GPU's logits (outside near ties) and the counters its update, bit for bit."""
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


def test_7b_decode_step_all_rows_both_paths():
    from continuous_batching_decode_gb300 import build
    build.build()
    B, lo, hi, seed = 32, 256, 4096, 0
    m = gu.Model("7b", max_rows=B, max_slots=B, mbps=(hi + 1 + 31) // 32)
    try:
        s = m.shape
        V = s["vocab"]
        db = synth.decode_batch(B, lo, hi, V, seed)
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
        rows = [(i, db["tokens"][i], ctx[i], 0, 1) for i in range(B)]
        samp = [dict(temperature=1.0, top_p=0.3, top_k=0, frequency_penalty=1.0, penalty_decay=0.996, seed=seed,
                     request_id=i, token_index=0) for i in range(B)]
        results = {}
        # path 1: cbd_step, launch by launch
        cv.zero_()
        toks, z_gpu = gu.run_step(m, pool, rows, tables, nbps, samp)
        results["cbd_step"] = (toks, z_gpu, cv.cpu().numpy())
        # path 2: the benchmark's path, a resident batch replayed as a graph
        b = cbd.batch_create(m.e, pool.p, rows, tables, nbps, samp)
        try:
            cbd.batch_set_graph(b, True)
            tok_d = torch.zeros(B, dtype=torch.int32, device="cuda")
            lg_d = torch.zeros(B, V, dtype=torch.float32, device="cuda")
            for _ in range(2):                   # capture + launch, then replay
                cv.zero_()
                cbd.batch_run(m.e, pool.p, b, tok_d, lg_d)
                cbd.engine_check(m.e)
            assert cbd.batch_captures(b) == 1
            results["graph replay"] = (tok_d.cpu().numpy(), lg_d.cpu().numpy().astype(np.float64),
                                       cv.cpu().numpy())
        finally:
            cbd.batch_destroy(b)
        # the oracle, 8 rows at a time (each decode row reads only its own
        # KV, so the rows are independent; this bounds the host memory the
        # fp64 KV copies take)
        om_ = m.oracle(cache=False)
        z = np.zeros((B, V))
        for g0 in range(0, B, 8):
            grp = list(range(g0, min(B, g0 + 8)))
            kv = gu.oracle_kv_from_gpu(m, pool, tables, {i: ctx[i] for i in grp})
            z[grp] = om.step(om_, kv, [(rows[i][0], rows[i][1], rows[i][2], 1) for i in grp])
            del kv
        pool.close()
        pre = np.zeros(V, np.float32)
        for path, (toks, zg, post) in results.items():
            mx, mean = gu.assert_logits_close(zg, z, f"7B step, {path}")
            print(f"7B step, {path}, all {B} rows: max-abs {mx:.3g} mean-abs {mean:.3g}")
            checked = 0
            for i in range(B):
                p = gu.sampling_params(samp[i])
                u = gu.uniform_of(samp[i])
                lf = zg[i].astype(np.float32)
                if not gu.sampling_near_tie(lf, pre, p, u):
                    assert toks[i] == osamp.sample_row(lf, pre, p, u), f"{path} row {i}"
                    checked += 1
                np.testing.assert_array_equal(post[i], osamp.update_counters(pre, int(toks[i]), 0.996))
            assert checked >= B - 2, f"{path}: only {checked} rows outside near ties"
    finally:
        m.close()
