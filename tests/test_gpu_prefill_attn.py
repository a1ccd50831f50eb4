"""GPU parity of the prefill attention kernel ("20.3 服务、批处理与流式"
section 20.3.2: a prompt chunk's rows are consecutive positions of one
sequence, so a block of them shares each K/V block it reads), over bf16 and
FP8 (E4M3) K/V.

Prefill runs (16+ rows of one slot at consecutive positions, in any row
order) take the kernel; other rows keep the streaming kernel.  The kernel computes the
streaming kernel's arithmetic (q and P split into bf16 hi + lo, exp2 softmax)
in another summation order, so: logits meet the oracle's tolerance with it on
and off, over runs that start at position 0 and runs that continue an
earlier prefix, runs that are not a multiple of the query block, a run of
exactly 16 rows, a 15-row run (which stays on the streaming kernel) and two
runs whose rows alternate in the row array; two runs are bit-identical, and
so is the step with its rows reversed; greedy ids agree outside near ties.
"""
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


def run_case(m, seed, with_kernel, reverse=False):
    """Slots 0-2 decode (contexts 9, 70, 200); slot 3 continues a 45-token
    prefix with 77 prompt rows; slot 4 brings a 16-row prompt, slot 5 a
    15-row one; slots 6 and 7 bring 18-row prompts whose rows alternate in
    the row array.  Returns tokens, logits, the rows and the prefixes."""
    V = m.shape["vocab"]
    rng = np.random.default_rng(seed)
    ctx = [9, 70, 200]
    pre3 = 45
    n_prompt = {3: 77, 4: 16, 5: 15, 6: 18, 7: 18}
    need = {s: (c + 1 + 31) // 32 for s, c in enumerate(ctx)}
    need.update({3: (pre3 + 77 + 31) // 32, 4: 1, 5: 1, 6: 1, 7: 1})
    n_pool = sum(need.values()) + 2
    tables, nbps = synth.permuted_tables(need, n_pool, 16, rng)
    pool = m.pool(n_pool)
    priors = {s: synth.random_tokens(rng, c, V) for s, c in enumerate(ctx)}
    priors[3] = synth.random_tokens(rng, pre3, V)
    cbd.engine_set_prefill_attention(m.e, with_kernel)
    for s, pr in priors.items():
        gu.gpu_prefill(m, pool, s, pr, tables, nbps, chunk=64)
    toks = synth.random_tokens(rng, 3, V)
    prompts = {s: synth.random_tokens(rng, n, V) for s, n in n_prompt.items()}
    start = {3: pre3, 4: 0, 5: 0, 6: 0, 7: 0}

    def row(s, i):
        n = n_prompt[s]
        return (s, prompts[s][i], start[s] + i, 1, 1 if i == n - 1 else 0)

    rows = [(s, toks[s], c, 0, 1) for s, c in enumerate(ctx)]
    for s in (3, 4, 5):
        rows += [row(s, i) for i in range(n_prompt[s])]
    for i in range(18):
        rows += [row(6, i), row(7, i)]
    if reverse:
        rows = rows[::-1]
    samp = [dict(GREEDY, request_id=k) for k in range(sum(1 for r in rows if r[4]))]
    got, z = gu.run_step(m, pool, rows, tables, nbps, samp)
    pool.close()
    return got, z, rows, priors


@pytest.mark.parametrize("kv_fp8", [False, True], ids=["bf16_kv", "e4m3_kv"])
@pytest.mark.parametrize("shape", ["tiny", "hd128"])
def test_prefill_kernel_matches_oracle(shape, kv_fp8):
    from continuous_batching_decode_gb300 import build
    build.build()
    m = gu.Model(shape, max_rows=256, max_slots=8, mbps=16, kv_fp8=kv_fp8)
    try:
        res = {}
        for on in (True, False):
            res[on] = run_case(m, 5, on)
        got2, z2, _, _ = run_case(m, 5, True)
        np.testing.assert_array_equal(z2, res[True][1])
        np.testing.assert_array_equal(got2, res[True][0])
        got3, z3, _, _ = run_case(m, 5, True, reverse=True)    # sampled rows come out reversed
        np.testing.assert_array_equal(z3[::-1], res[True][1])
        np.testing.assert_array_equal(got3[::-1], res[True][0])
        _, _, rows, priors = res[True]
        om_ = m.oracle()
        kv = {s: om.SequenceKV(om_.cfg, 256) for s in range(8)}
        for s, pr in priors.items():
            om.prefill(om_, kv, s, pr)
        z = om.step(om_, kv, [(r[0], r[1], r[2], r[4]) for r in rows])
        for on, (got, zg, _, _) in res.items():
            gu.assert_logits_close(zg, z, f"{shape} ({'e4m3' if kv_fp8 else 'bf16'} KV) prefill runs, "
                                          f"prefill kernel {'on' if on else 'off'}")
            for j in range(len(z)):
                if not gu.greedy_near_tie(z[j]):
                    assert got[j] == int(np.argmax(z[j])), f"kernel {on}: row {j}"
    finally:
        cbd.engine_set_prefill_attention(m.e, True)
        m.close()
