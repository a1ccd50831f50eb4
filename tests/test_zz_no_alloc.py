"""The allocation-free sampler entry point (cbd_sample_static).

Callers that cannot allocate device memory -- a framework whose caching
allocator already holds the device's memory budget, or a serving loop that
forbids allocation after warm-up -- use cbd_sample_static, whose scratch is
a fixed-size array inside libcbd.  This test drives it through the C ABI and
checks, over two calls in a row, that it returns exactly what the engine's
cbd_sample returns on copies of the same logits and counters: the same
token ids and the same updated counters (the sampler's bar is bit-exact).
The ids and counters are also held to the oracle sampler on the same logits,
counters and uniforms, outside near ties.  The array's error word stays
clear on these inputs; a row whose logits are all -inf has nothing to draw,
which the check call reports once and then clears.  The size limits are
checked too.  The file is named to be collected last."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import continuous_batching_decode_gb300 as cbd
    from continuous_batching_decode_gb300 import build, synth
    from oracle import sampler as osamp
    from tests import gpu_util as gu


@pytest.mark.parametrize("vocab_shape", ["tiny", "7b"])
def test_static_sampler_matches_engine_sampler(vocab_shape):
    build.build()
    shape = synth.MODEL_SHAPES["tiny"]
    V = synth.MODEL_SHAPES[vocab_shape]["vocab"]
    shape = dict(shape, vocab=V)
    w = synth.make_weights(shape, seed=0, device="cuda")
    e = cbd.engine_create(cbd.make_config(shape, 16, 16, 4), w)
    try:
        rng = np.random.default_rng(17)
        m = 12
        slots = [int(s) for s in rng.permutation(16)[:m]]
        engine_cnt = cbd.device_view(cbd.engine_counters(e), (16, V), "f32")
        c0 = np.where(rng.random((16, V)) < 0.05, rng.integers(1, 5, (16, V)), 0).astype(np.float32)
        engine_cnt.copy_(torch.from_numpy(c0).cuda())
        own_cnt = torch.from_numpy(c0.copy()).cuda()
        configs = [dict(temperature=0.0, frequency_penalty=1.0, penalty_decay=0.996),
                   dict(temperature=1.0, top_p=0.3, frequency_penalty=1.0, penalty_decay=0.996),
                   dict(temperature=0.8, top_p=0.9, top_k=40, presence_penalty=0.5, penalty_decay=0.99)]
        cbd.sample_static_check()           # start from a clear error word
        checked = 0
        for call in range(2):
            pre = own_cnt.cpu().numpy().copy()
            lg_np = rng.normal(0, 2.0, (m, V)).astype(np.float32)
            lg = torch.from_numpy(lg_np).cuda()
            samp = [dict(configs[j % 3], seed=5, request_id=900 + j, token_index=call) for j in range(m)]
            us = None if call == 0 else [float(u) for u in rng.random(m)]
            a = torch.full((m,), -1, dtype=torch.int32, device="cuda")
            b = torch.full((m,), -1, dtype=torch.int32, device="cuda")
            cbd.sample(e, lg, slots, samp, us, a)
            cbd.sample_static(lg, own_cnt, slots, samp, us, b)
            torch.cuda.synchronize()
            ta, tb = a.cpu().numpy(), b.cpu().numpy()
            np.testing.assert_array_equal(ta, tb)
            post = own_cnt.cpu().numpy()
            np.testing.assert_array_equal(engine_cnt.cpu().numpy(), post)
            assert (tb >= 0).all()
            cbd.sample_static_check()       # no row lacked a token
            # the oracle sampler on the same logits, counters and uniforms
            for j, s in enumerate(slots):
                p = gu.sampling_params(samp[j])
                u = us[j] if us is not None else gu.uniform_of(samp[j])
                np.testing.assert_array_equal(post[s], osamp.update_counters(pre[s], int(tb[j]), p.penalty_decay))
                if gu.sampling_near_tie(lg_np[j], pre[s], p, u):
                    continue
                assert int(tb[j]) == osamp.sample_row(lg_np[j], pre[s], p, u), f"call {call} row {j}"
                checked += 1
        assert checked >= 20
        # a row whose logits are all -inf (every id masked) has no token to
        # draw: it gets token 0, the error word records it, the check call
        # reports it once and clears it
        lg = torch.from_numpy(rng.normal(0, 2.0, (2, V)).astype(np.float32)).cuda()
        lg[1] = float("-inf")
        out = torch.full((2,), -1, dtype=torch.int32, device="cuda")
        samp = [dict(temperature=1.0, top_p=0.9, seed=1, request_id=1),
                dict(temperature=1.0, top_p=0.9, seed=1, request_id=2)]
        cbd.sample_static(lg, own_cnt, [0, 1], samp, None, out)
        with pytest.raises(cbd.CbdError) as ei:
            cbd.sample_static_check()
        assert ei.value.status == cbd.EDEVICE and "no token" in str(ei.value)
        assert int(out.cpu()[1]) == 0 and int(out.cpu()[0]) >= 0
        cbd.sample_static_check()           # cleared by the previous check
        with pytest.raises(cbd.CbdError) as ei:
            big = torch.zeros(cbd.SAMPLE_STATIC_MAX_ROWS + 1, V, device="cuda")
            out = torch.zeros(cbd.SAMPLE_STATIC_MAX_ROWS + 1, dtype=torch.int32, device="cuda")
            cbd.sample_static(big, own_cnt, list(range(cbd.SAMPLE_STATIC_MAX_ROWS + 1)),
                              [dict(temperature=0.0)] * (cbd.SAMPLE_STATIC_MAX_ROWS + 1), None, out)
        assert ei.value.status == cbd.EINVAL and "static scratch" in str(ei.value)
    finally:
        cbd.engine_destroy(e)
