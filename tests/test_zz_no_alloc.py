"""The allocation-free sampler entry point (cbd_sample_static).

Callers that cannot allocate device memory -- a framework whose caching
allocator already holds the device's memory budget, or a serving loop that
forbids allocation after warm-up -- use cbd_sample_static, whose scratch is
a fixed-size array inside libcbd.  This test drives it through the C ABI and
checks, over two calls in a row, that it returns exactly what the engine's
cbd_sample returns on copies of the same logits and counters: the same
token ids and the same updated counters (the sampler's bar is bit-exact).
It also checks the size limits.  The file is named to be collected last."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import continuous_batching_decode_gb300 as cbd
    from continuous_batching_decode_gb300 import build, synth


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
        for call in range(2):
            lg = torch.from_numpy(rng.normal(0, 2.0, (m, V)).astype(np.float32)).cuda()
            samp = [dict(configs[j % 3], seed=5, request_id=900 + j, token_index=call) for j in range(m)]
            us = None if call == 0 else [float(u) for u in rng.random(m)]
            a = torch.full((m,), -1, dtype=torch.int32, device="cuda")
            b = torch.full((m,), -1, dtype=torch.int32, device="cuda")
            cbd.sample(e, lg, slots, samp, us, a)
            cbd.sample_static(lg, own_cnt, slots, samp, us, b)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(a.cpu().numpy(), b.cpu().numpy())
            np.testing.assert_array_equal(engine_cnt.cpu().numpy(), own_cnt.cpu().numpy())
            assert (a >= 0).all()
        with pytest.raises(cbd.CbdError) as ei:
            big = torch.zeros(cbd.SAMPLE_STATIC_MAX_ROWS + 1, V, device="cuda")
            out = torch.zeros(cbd.SAMPLE_STATIC_MAX_ROWS + 1, dtype=torch.int32, device="cuda")
            cbd.sample_static(big, own_cnt, list(range(cbd.SAMPLE_STATIC_MAX_ROWS + 1)),
                              [dict(temperature=0.0)] * (cbd.SAMPLE_STATIC_MAX_ROWS + 1), None, out)
        assert ei.value.status == cbd.EINVAL and "static scratch" in str(ei.value)
    finally:
        cbd.engine_destroy(e)
