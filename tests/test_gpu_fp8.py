"""GPU parity with an FP8 (E4M3) KV pool ("大模型推理为什么需要 Continuous
Batching", section 6: KV quantised to FP8 to fit more sequences).

The oracle stores K and V rounded to E4M3 (round to nearest even, saturating;
oracle/model.py, pinned against the format's bit definition) and otherwise
computes in fp64.  Bars: the same logit tolerance as bf16 KV; the pool holds
exactly E4M3 values that match the oracle's rounding up to a rounding-boundary
neighbour; paging and row order stay bit-exact; the pool takes half the bytes.
"""
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
    from tests.test_gpu_step import preload_counters, tiny_setup


@pytest.fixture(scope="module", params=[0, 1, 2], ids=["auto", "gemv", "tcgen05"])
def tiny8(request):
    """The tiny decoder over an FP8 KV pool, each GEMM path (the K/V stores
    sit in the GEMV's and the tensor-core GEMM's epilogues)."""
    from continuous_batching_decode_gb300 import build
    build.build()
    m = gu.Model("tiny", max_rows=512, max_slots=8, mbps=16, kv_fp8=True)
    cbd.engine_set_gemm_path(m.e, request.param)
    m.attn_path = 0
    yield m
    m.close()


def e4m3_step(x):
    """Spacing of E4M3 values at |x| (for one-neighbour tolerances)."""
    a = np.maximum(np.abs(x), 2.0 ** -9)
    _, e = np.frexp(a)
    return np.ldexp(1.0, np.maximum(e - 4, -9))


def test_fp8_tiny_step_matches_oracle(tiny8):
    wl, pool, tables, nbps, rows, sampling = tiny_setup(tiny8, 1)
    cv, c4 = preload_counters(tiny8, wl)
    pre = cv.cpu().numpy().copy()
    toks, z_gpu = gu.run_step(tiny8, pool, rows, tables, nbps, sampling)
    post = cv.cpu().numpy()
    om_ = tiny8.oracle()
    kv = {s: om.SequenceKV(om_.cfg, 128) for s in range(5)}
    for s, prior in enumerate(wl["prior"]):
        om.prefill(om_, kv, s, prior)
    z = om.step(om_, kv, [(r[0], r[1], r[2], r[4]) for r in rows])
    gu.assert_logits_close(z_gpu, z, "tiny FP8-KV step")
    for j in range(4):
        if not gu.greedy_near_tie(z[j]):
            assert toks[j] == int(np.argmax(osamp.penalize(z_gpu[j].astype(np.float32), pre[j], 0.0, 1.0)))
    for j in range(5):
        p = gu.sampling_params(sampling[j])
        np.testing.assert_array_equal(post[j], osamp.update_counters(pre[j], int(toks[j]), p.penalty_decay))
    # the pool holds E4M3 values; layer 0's equal the oracle's rounding up to
    # a rounding-boundary neighbour (fp32 vs fp64 inputs to the rounding)
    for s, c in enumerate(wl["contexts"] + [39]):
        n = c + 1
        K, V = pool.gather(tables, s, n)
        for l in range(om_.cfg.n_layers):
            for A, B in ((K[l], kv[s].K[l][:n]), (V[l], kv[s].V[l][:n])):
                np.testing.assert_array_equal(om.round_to_e4m3(A), A)
                if l == 0:
                    assert np.mean(A != B) < 0.01, f"slot {s}: {np.mean(A != B):.3%} entries differ"
                    assert (np.abs(A - B) <= e4m3_step(B) * 1.0001).all()
    # over the GPU's own KV only the step's arithmetic differs
    prior = {s: c for s, c in enumerate(wl["contexts"])}
    kv2 = gu.oracle_kv_from_gpu(tiny8, pool, tables, prior)
    kv2[4] = om.SequenceKV(om_.cfg, 64)
    z2 = om.step(om_, kv2, [(r[0], r[1], r[2], r[4]) for r in rows])
    err2 = np.abs(z_gpu - z2)
    assert err2.mean() <= 2e-4 and err2.max() <= 2e-3 * np.abs(z2).max(), (err2.mean(), err2.max())
    pool.close()


def test_fp8_paging_and_row_order_are_bit_exact(tiny8):
    outs = []
    for placement in (1, 2):
        wl, pool, tables, nbps, rows, sampling = tiny_setup(tiny8, placement)
        preload_counters(tiny8, wl)
        toks, z = gu.run_step(tiny8, pool, rows, tables, nbps, sampling)
        K0, V0 = pool.gather(tables, 3, 65)
        outs.append((toks, z, K0[1], V0[1]))
        if placement == 2:    # same placement, rows reversed
            preload_counters(tiny8, wl)
            samp_r = [sampling[4]] + sampling[:4][::-1]
            toks_r, z_r = gu.run_step(tiny8, pool, rows[::-1], tables, nbps, samp_r)
            order = [4, 3, 2, 1, 0]
            np.testing.assert_array_equal(z_r[order], z)
            np.testing.assert_array_equal(toks_r[order], toks)
        pool.close()
    for i in range(4):
        np.testing.assert_array_equal(outs[0][i], outs[1][i])


def test_fp8_pool_is_half_the_bytes(tiny8):
    p8 = cbd.kv_pool_create(tiny8.e, 10)
    m16 = gu.Model("tiny", max_rows=16, max_slots=2, mbps=4)
    p16 = cbd.kv_pool_create(m16.e, 10)
    try:
        assert cbd.kv_pool_data(p8)[1] * 2 == cbd.kv_pool_data(p16)[1]
        with pytest.raises(cbd.CbdError):
            cbd.engine_set_attention_path(tiny8.e, 1)        # FP8 KV runs on the streaming kernel only
    finally:
        cbd.kv_pool_destroy(p8)
        cbd.kv_pool_destroy(p16)
        m16.close()
