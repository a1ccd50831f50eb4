"""Pins for the fp64 decoder oracle (CPU only).

Each check fixes the oracle to something other than itself: a scalar-loop
brute force on a hand-sized model, closed forms of RMSNorm / RoPE /
attention, a hand-worked RoPE example, and the invariants the pages state
(batching and chunking leave results unchanged).  The mutation tests at the
end plant plausible mistakes in the oracle and check that a pin catches each.
"""
import math
import os

import numpy as np
import pytest

from oracle import model as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_exact(rng, shape, std=0.3):
    """Random values that are exactly representable in bf16."""
    return om.round_to_bf16(rng.normal(0, std, size=shape))


def small_model(seed=0, L=2, d=8, hq=2, hkv=1, hd=4, F=12, V=16, std=0.3):
    rng = np.random.default_rng(seed)
    cfg = om.ModelConfig(L, d, hq, hkv, hd, F, V)
    w = {"embed": bf16_exact(rng, (V, d), 1.0), "lm_head": bf16_exact(rng, (V, d), std),
         "final_norm": bf16_exact(rng, (d,), 0.5) + 1.0}
    for l in range(L):
        w[f"{l}.attn_norm"] = om.round_to_bf16(1.0 + rng.normal(0, 0.2, d))
        w[f"{l}.ffn_norm"] = om.round_to_bf16(1.0 + rng.normal(0, 0.2, d))
        w[f"{l}.wq"] = bf16_exact(rng, (hq * hd, d), std)
        w[f"{l}.wk"] = bf16_exact(rng, (hkv * hd, d), std)
        w[f"{l}.wv"] = bf16_exact(rng, (hkv * hd, d), std)
        w[f"{l}.wo"] = bf16_exact(rng, (d, hq * hd), std)
        w[f"{l}.w_gate"] = bf16_exact(rng, (F, d), std)
        w[f"{l}.w_up"] = bf16_exact(rng, (F, d), std)
        w[f"{l}.w_down"] = bf16_exact(rng, (d, F), std)
    return cfg, w


# ---------------------------------------------------------------- brute force
def brute_logits(cfg, w, seqs):
    """Scalar loops written from the definition: each sequence processed token
    by token, KV in Python lists, softmax by explicit sums.  seqs: list of
    token lists.  Returns the last token's logits of each sequence."""
    d, hq, hkv, hd, F = cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim
    out = []

    def rms(v, g):
        ms = sum(a * a for a in v) / len(v)
        r = 1.0 / math.sqrt(ms + cfg.rms_eps)
        return [a * r * gg for a, gg in zip(v, g)]

    def matvec(W, v):
        return [sum(W[i][j] * v[j] for j in range(len(v))) for i in range(len(W))]

    def bf(v):
        return [float(om.round_to_bf16(np.float64(a))) for a in v]

    for toks in seqs:
        K = [[] for _ in range(cfg.n_layers)]
        Vv = [[] for _ in range(cfg.n_layers)]
        last = None
        for p, t in enumerate(toks):
            x = [float(a) for a in w["embed"][t]]
            for l in range(cfg.n_layers):
                h = rms(x, w[f"{l}.attn_norm"])
                q = matvec(w[f"{l}.wq"], h)
                k = matvec(w[f"{l}.wk"], h)
                v = matvec(w[f"{l}.wv"], h)
                for heads, vec in ((hq, q), (hkv, k)):
                    for hh in range(heads):
                        base = hh * hd
                        for i in range(hd // 2):
                            ang = p * cfg.rope_base ** (-2.0 * i / hd)
                            a, b = vec[base + i], vec[base + i + hd // 2]
                            vec[base + i] = a * math.cos(ang) - b * math.sin(ang)
                            vec[base + i + hd // 2] = b * math.cos(ang) + a * math.sin(ang)
                K[l].append(bf(k))
                Vv[l].append(bf(v))
                o = []
                for hh in range(hq):
                    g = hh // (hq // hkv)
                    sc = []
                    for j in range(p + 1):
                        sc.append(sum(q[hh * hd + e] * K[l][j][g * hd + e] for e in range(hd)) / math.sqrt(hd))
                    m = max(sc)
                    ex = [math.exp(s - m) for s in sc]
                    tot = sum(ex)
                    for e in range(hd):
                        o.append(sum(ex[j] / tot * Vv[l][j][g * hd + e] for j in range(p + 1)))
                att = matvec(w[f"{l}.wo"], o)
                x = [a + b for a, b in zip(x, att)]
                h = rms(x, w[f"{l}.ffn_norm"])
                gt = matvec(w[f"{l}.w_gate"], h)
                up = matvec(w[f"{l}.w_up"], h)
                a_ = [gg / (1.0 + math.exp(-gg)) * uu for gg, uu in zip(gt, up)]
                dn = matvec(w[f"{l}.w_down"], a_)
                x = [a + b for a, b in zip(x, dn)]
            last = matvec(w["lm_head"], rms(x, w["final_norm"]))
        out.append(last)
    return np.array(out)


def oracle_batched(cfg, w, seqs):
    """Prefill all sequences except their last token, then one batched step
    with every sequence's last token as a decode row."""
    m = om.OracleModel(cfg, w)
    kv = {s: om.SequenceKV(cfg, 4) for s in range(len(seqs))}
    for s, toks in enumerate(seqs):
        if len(toks) > 1:
            om.prefill(m, kv, s, toks[:-1])
    rows = [(s, toks[-1], len(toks) - 1, 1) for s, toks in enumerate(seqs)]
    return om.step(m, kv, rows)


def test_brute_force_small_model():
    cfg, w = small_model()
    seqs = [[3], [1, 4, 1, 5, 9], [2, 6, 5, 3, 5, 8, 9, 7]]
    ref = brute_logits(cfg, w, seqs)
    got = oracle_batched(cfg, w, seqs)
    assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_brute_force_gqa_group_of_two():
    cfg, w = small_model(seed=3, hq=4, hkv=2, hd=4, d=8)
    seqs = [[7, 7, 2], [0, 15, 8, 8, 1, 2]]
    ref = brute_logits(cfg, w, seqs)
    got = oracle_batched(cfg, w, seqs)
    assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


# ----------------------------------------------------------- closed forms
def test_rmsnorm_constant_vector():
    g = np.array([1.0, 2.0, -0.5, 4.0])
    for c in (3.0, -0.25):
        out = om.rmsnorm(np.full(4, c), g, 1e-6)
        np.testing.assert_allclose(out, g * c / math.sqrt(c * c + 1e-6), rtol=1e-15)


def test_rope_identity_at_zero():
    x = np.random.default_rng(1).normal(size=(3, 2, 8))
    np.testing.assert_array_equal(om.rope(x, np.zeros(3, dtype=int), 10000.0), x)


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(2)
    x = rng.normal(size=(5, 3, 16))
    y = om.rope(x, rng.integers(0, 5000, 5), 10000.0)
    nx = x[..., :8] ** 2 + x[..., 8:] ** 2
    ny = y[..., :8] ** 2 + y[..., 8:] ** 2
    np.testing.assert_allclose(ny, nx, rtol=1e-12)


def test_rope_relative_position():
    """q(p+D) . k(p'+D) == q(p) . k(p') for any shift D."""
    rng = np.random.default_rng(3)
    q, k = rng.normal(size=(1, 1, 64)), rng.normal(size=(1, 1, 64))
    for p, pp, D in ((5, 2, 100), (0, 37, 4096), (900, 899, 7)):
        a = np.sum(om.rope(q, [p + D], 1e4) * om.rope(k, [pp + D], 1e4))
        b = np.sum(om.rope(q, [p], 1e4) * om.rope(k, [pp], 1e4))
        assert abs(a - b) <= 1e-11 * max(1.0, abs(b))


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, *v = line.split()
            vals[k] = [float(a) for a in v]
    return vals


def test_rope_hand_worked_example():
    g = read_golden("rope_hd4_p1.txt")
    x = np.array(g["x"]).reshape(1, 1, 4)
    y = om.rope(x, [int(g["pos"][0])], g["base"][0]).reshape(-1)
    np.testing.assert_allclose(y, g["out"], rtol=0, atol=1e-15)


def test_attention_single_position_returns_v():
    rng = np.random.default_rng(4)
    q = rng.normal(size=(4, 8))
    K, V = rng.normal(size=(1, 2, 8)), rng.normal(size=(1, 2, 8))
    o = om.attend(q, K, V)
    np.testing.assert_array_equal(o, np.repeat(V[0], 2, axis=0))


def test_attention_equal_keys_average_values():
    """Identical keys give uniform weights: output = mean of the values."""
    rng = np.random.default_rng(5)
    q = rng.normal(size=(2, 8))
    K = np.repeat(rng.normal(size=(1, 1, 8)), 6, axis=0)
    V = rng.normal(size=(6, 1, 8))
    np.testing.assert_allclose(om.attend(q, K, V), np.repeat(V.mean(0), 2, axis=0), rtol=1e-13)


def test_gqa_with_equal_heads_is_mha():
    """H_kv == H_q: head i reads KV head i (explicit per-head loop)."""
    rng = np.random.default_rng(6)
    q = rng.normal(size=(3, 8))
    K, V = rng.normal(size=(5, 3, 8)), rng.normal(size=(5, 3, 8))
    o = om.attend(q, K, V)
    for i in range(3):
        s = K[:, i, :] @ q[i] / math.sqrt(8)
        p = np.exp(s - s.max())
        p /= p.sum()
        np.testing.assert_allclose(o[i], p @ V[:, i, :], rtol=1e-13)


def test_bf16_rounding_ties_to_even_and_matches_torch():
    one = 1.0
    assert om.round_to_bf16(one + 2 ** -8) == 1.0                 # tie -> even (1.0)
    assert om.round_to_bf16(one + 3 * 2 ** -8) == one + 2 ** -6   # tie -> even mantissa
    assert om.round_to_bf16(one + 2 ** -8 + 2 ** -20) == one + 2 ** -7
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(7).normal(0, 3, size=10000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(om.round_to_bf16(x.astype(np.float64)), ref)


def e4m3_code_value(code: int) -> float:
    """Value of an FP8 E4M3 bit pattern, straight from the format: sign bit,
    exponent field E (4 bits, bias 7), fraction F (3 bits); E == 0 is
    subnormal (F/8 * 2^-6); E == 15 with F == 7 is NaN; no infinities."""
    sgn = -1.0 if code & 0x80 else 1.0
    E, F = (code >> 3) & 0xF, code & 7
    if E == 15 and F == 7:
        return math.nan
    if E == 0:
        return sgn * F / 8 * 2.0 ** -6
    return sgn * (1 + F / 8) * 2.0 ** (E - 7)


def test_e4m3_rounding_against_the_format():
    finite = sorted({e4m3_code_value(c) for c in range(256) if not math.isnan(e4m3_code_value(c))})
    assert len(finite) == 253 and finite[-1] == 448.0 and finite[0] == -448.0   # +-0 collapse
    vals = np.array(finite)
    np.testing.assert_array_equal(om.round_to_e4m3(vals), vals)         # representable: unchanged
    pos = [v for v in finite if v >= 0]
    code_of = {e4m3_code_value(c): c for c in range(128)}
    for lo, hi in zip(pos, pos[1:]):
        mid = (lo + hi) / 2
        even = lo if code_of[lo] % 2 == 0 else hi                          # ties to the even code
        assert om.round_to_e4m3(mid) == even, (lo, hi)
        assert om.round_to_e4m3(mid - (hi - lo) * 1e-6) == lo
        assert om.round_to_e4m3(mid + (hi - lo) * 1e-6) == hi
        assert om.round_to_e4m3(-mid) == -even
    assert om.round_to_e4m3(470.0) == 448.0 and om.round_to_e4m3(1e9) == 448.0   # saturation
    assert om.round_to_e4m3(-1e9) == -448.0
    assert om.round_to_e4m3(2.0 ** -10) == 0.0 and om.round_to_e4m3(2.0 ** -10 + 1e-12) == 2.0 ** -9
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    x = np.random.default_rng(8).normal(0, 40, size=20000)
    x = x[np.abs(x) <= 440]
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(om.round_to_e4m3(x.astype(np.float32).astype(np.float64)), ref)


def test_e4m3_kv_format_rounds_stored_kv():
    cfg, w = small_model(seed=3)
    rows = [(0, 3, 0, 1), (0, 5, 1, 1)]
    kv = {0: om.SequenceKV(cfg, 4)}
    om.step(om.OracleModel(cfg, w, kv_format="e4m3"), kv, rows)
    for l in range(cfg.n_layers):
        K = kv[0].K[l][:2]
        np.testing.assert_array_equal(om.round_to_e4m3(K), K)
    kv_b = {0: om.SequenceKV(cfg, 4)}
    om.step(om.OracleModel(cfg, w), kv_b, rows)
    assert np.abs(kv_b[0].K[0][:2] - kv[0].K[0][:2]).max() > 0      # a different rounding is used
    with pytest.raises(ValueError):
        om.OracleModel(cfg, w, kv_format="fp16")


# ------------------------------------------------------------- invariants
def tiny_model(seed=0):
    from continuous_batching_decode_gb300 import synth
    s = synth.MODEL_SHAPES["tiny"]
    w = {k: synth.bf16_bits(v) for k, v in synth.make_weights(s, seed).items()}
    return om.ModelConfig(**s), w


@pytest.fixture(scope="module")
def tiny():
    return tiny_model()


def test_batched_step_equals_independent_rows(tiny):
    """Batching must not change results (page 14-1, section 3): one step over
    a mixed row set equals the same rows run one at a time."""
    cfg, w = tiny
    m = om.OracleModel(cfg, w)
    rng = np.random.default_rng(11)
    ctx = [5, 17, 33]
    toks = [list(rng.integers(0, cfg.vocab, c + 1)) for c in ctx]
    prompt = list(rng.integers(0, cfg.vocab, 12))

    def fresh():
        kv = {s: om.SequenceKV(cfg, 8) for s in range(4)}
        for s, t in enumerate(toks):
            om.prefill(m, kv, s, t[:-1])
        return kv

    kv_a = fresh()
    rows = [(s, t[-1], ctx[s], 1) for s, t in enumerate(toks)]
    rows += [(3, prompt[i], i, 1 if i == 11 else 0) for i in range(12)]
    za = om.step(m, kv_a, rows)
    kv_b = fresh()
    zb = []
    for r in rows:                       # one row per step, prompt rows in order
        out = om.step(m, kv_b, [r])
        if r[3]:
            zb.append(out[0])
    zb = np.array(zb)
    assert np.max(np.abs(za - zb)) <= 1e-12 * np.max(np.abs(zb))
    for s in range(4):
        n = kv_a[s].length
        for l in range(cfg.n_layers):
            np.testing.assert_array_equal(kv_a[s].K[l][:n], kv_b[s].K[l][:n])


def test_row_order_does_not_matter(tiny):
    cfg, w = tiny
    m = om.OracleModel(cfg, w)
    rng = np.random.default_rng(12)
    prompt = list(rng.integers(0, cfg.vocab, 9))
    rows = [(0, prompt[i], i, 1 if i == 8 else 0) for i in range(9)]
    za = om.step(m, {0: om.SequenceKV(cfg, 8)}, rows)
    zb = om.step(m, {0: om.SequenceKV(cfg, 8)}, rows[::-1])
    np.testing.assert_allclose(za, zb, rtol=0, atol=1e-12)


def test_chunked_prefill_equivalence(tiny):
    """One chunk == 8-token chunks == token by token (causal masking inside
    a chunk)."""
    cfg, w = tiny
    m = om.OracleModel(cfg, w)
    prompt = list(np.random.default_rng(13).integers(0, cfg.vocab, 40))
    outs, kvs = [], []
    for chunk in (None, 8, 1):
        kv = {0: om.SequenceKV(cfg, 64)}
        outs.append(om.prefill(m, kv, 0, prompt, chunk=chunk))
        kvs.append(kv[0])
    for z in outs[1:]:
        assert np.max(np.abs(z - outs[0])) <= 1e-12 * np.max(np.abs(outs[0]))
    for kv in kvs[1:]:
        for l in range(cfg.n_layers):
            np.testing.assert_array_equal(kv.K[l][:40], kvs[0].K[l][:40])
            np.testing.assert_array_equal(kv.V[l][:40], kvs[0].V[l][:40])


# ---------------------------------------------------------------- mutations
def _mutations():
    good_rope = om.rope

    def rope_sign(x, pos, base):
        return good_rope(x, -np.asarray(pos), base)

    def rope_interleaved(x, pos, base):
        hd = x.shape[-1]
        perm = np.concatenate([np.arange(0, hd, 2), np.arange(1, hd, 2)])
        inv = np.argsort(perm)
        return good_rope(x[..., perm], pos, base)[..., inv]

    good_attend = om.attend

    def attend_no_scale(q, K, V):
        return good_attend(q * math.sqrt(q.shape[-1]), K, V)

    def attend_wrong_group(q, K, V):
        hq, hkv = q.shape[0], K.shape[1]
        if hkv == 1:
            return good_attend(q, K, V)
        idx = np.arange(hq) % hkv          # interleaved instead of contiguous groups
        return np.stack([good_attend(q[i:i + 1], K[:, idx[i]:idx[i] + 1], V[:, idx[i]:idx[i] + 1])[0]
                         for i in range(hq)])

    good_rms = om.rmsnorm

    def rms_no_eps_mean(x, g, eps):
        return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps) * g

    def silu_wrong(x):
        return x / (1.0 + np.exp(x))

    return [("rope", rope_sign), ("rope", rope_interleaved), ("attend", attend_no_scale),
            ("attend", attend_wrong_group), ("rmsnorm", rms_no_eps_mean), ("silu", silu_wrong)]


@pytest.mark.parametrize("idx", range(6))
def test_planted_mistakes_are_caught(idx, monkeypatch):
    name, bad = _mutations()[idx]
    monkeypatch.setattr(om, name, bad)
    cfg, w = small_model(seed=3, hq=4, hkv=2, hd=4, d=8)
    seqs = [[7, 7, 2], [0, 15, 8, 8, 1, 2]]
    caught = False
    try:
        test_rope_hand_worked_example()
    except AssertionError:
        caught = True
    got = oracle_batched(cfg, w, seqs)
    monkeypatch.undo()
    ref = brute_logits(cfg, w, seqs)
    caught = caught or np.max(np.abs(got - ref)) > 1e-9
    assert caught, f"mutation of {name} not caught"
