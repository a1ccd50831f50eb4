"""GPU: decode rows whose token is CBD_TOKEN_LAST read the token the engine's
sampler last drew for their slot ("20.3 服务、批处理与流式" section 20.3.2:
an iteration's inputs are the previous iteration's outputs), so a decode loop
can enqueue the next step before the tokens reach the host.

A step with CBD_TOKEN_LAST must equal, bit for bit (logits, drawn ids, the
K/V it appends), the same step with the previous step's ids passed
explicitly -- through cbd_step and through a resident batch replayed as a
graph; cbd_slot_reset resets a slot's last token to 0; prefill rows may not
use it."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import continuous_batching_decode_gb300 as cbd
    from tests import gpu_util as gu
    from tests.test_gpu_step import tiny_setup


def test_token_last_equals_explicit_previous_tokens():
    from continuous_batching_decode_gb300 import build
    build.build()
    m = gu.Model("tiny", max_rows=64, max_slots=8, mbps=16)
    try:
        wl, pool, tables, nbps, rows, sampling = tiny_setup(m, 1)
        ctx = wl["contexts"]
        samp = [dict(temperature=1.0, top_p=0.9, frequency_penalty=0.5, penalty_decay=0.99, seed=7,
                     request_id=100 + s, token_index=0) for s in range(4)]
        cv = gu.counters_view(m)
        cv.zero_()
        kv_pre, c_pre = pool.view.clone(), cv.clone()
        step1 = [(s, rows[s][1], ctx[s], 0, 1) for s in range(4)]

        def replay_step1():
            pool.view.copy_(kv_pre)
            cv.copy_(c_pre)
            t, _ = gu.run_step(m, pool, step1, tables, nbps, samp)
            return t

        t1 = replay_step1()
        samp2 = [dict(s, token_index=1) for s in samp]
        kv0, c0 = pool.view.clone(), cv.clone()
        # (b) CBD_TOKEN_LAST right after step 1: the ids it drew, read on the device
        tb, zb = gu.run_step(m, pool, [(s, cbd.TOKEN_LAST, ctx[s] + 1, 0, 1) for s in range(4)], tables, nbps,
                             samp2)
        kvb, cb = pool.view.clone(), cv.clone()
        # (a) explicit ids, from the same state
        pool.view.copy_(kv0)
        cv.copy_(c0)
        ta, za = gu.run_step(m, pool, [(s, int(t1[s]), ctx[s] + 1, 0, 1) for s in range(4)], tables, nbps, samp2)
        np.testing.assert_array_equal(zb, za)
        np.testing.assert_array_equal(tb, ta)
        assert torch.equal(pool.view, kvb) and torch.equal(cv, cb)
        # (c) the same through a resident batch replayed as a graph (step 1
        # replayed before each run, so the slots' last tokens are t1 again)
        b = cbd.batch_create(m.e, pool.p, [(s, cbd.TOKEN_LAST, ctx[s] + 1, 0, 1) for s in range(4)], tables, nbps,
                             samp2)
        try:
            cbd.batch_set_graph(b, True)
            for it in range(2):
                np.testing.assert_array_equal(replay_step1(), t1)
                tok_d = torch.zeros(4, dtype=torch.int32, device="cuda")
                lg_d = torch.zeros(4, m.shape["vocab"], dtype=torch.float32, device="cuda")
                cbd.batch_run(m.e, pool.p, b, tok_d, lg_d)
                cbd.engine_check(m.e)
                np.testing.assert_array_equal(lg_d.cpu().numpy().astype(np.float64), za)
                np.testing.assert_array_equal(tok_d.cpu().numpy(), ta)
        finally:
            cbd.batch_destroy(b)
        # (d) after a slot reset the slot's last token is 0
        pool.view.copy_(kv0)
        cv.copy_(c0)
        cbd.slot_reset(m.e, 2)
        cv.copy_(c0)
        _, zr = gu.run_step(m, pool, [(2, cbd.TOKEN_LAST, ctx[2] + 1, 0, 1)], tables, nbps, samp2[2:3])
        pool.view.copy_(kv0)
        cv.copy_(c0)
        _, ze = gu.run_step(m, pool, [(2, 0, ctx[2] + 1, 0, 1)], tables, nbps, samp2[2:3])
        np.testing.assert_array_equal(zr, ze)
        # (e) not on prefill rows
        with pytest.raises(cbd.CbdError):
            gu.run_step(m, pool, [(2, cbd.TOKEN_LAST, ctx[2] + 1, 1, 1)], tables, nbps, samp2[2:3])
        pool.close()
    finally:
        m.close()
