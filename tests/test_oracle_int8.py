"""Pins for the oracle's int8 weight quantisation (CPU only).

The pages name int8 weights ("RWKV Runner Albatross 后端", 边界与后续路线) and
no scheme; the reading is weight-only, symmetric, one fp32 scale per output
row: s = fp32(max|w| / 127), q = nearest integer to w / s (ties to even),
clamped to +-127.  These checks hold the oracle's vectorised code to that
definition by other means: exact rational arithmetic (fractions.Fraction)
for the scale and for every q, the invariants the definition implies, and a
hand-worked row."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import model as om


def exact_fp32_nearest(x: Fraction) -> float:
    """The fp32 value nearest to the rational x (ties to even), by search
    over the neighbours of numpy's candidate."""
    c = np.float32(float(x))
    best = None
    for cand in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        d = abs(Fraction(float(cand)) - x)
        key = (d, int(np.frombuffer(np.float32(cand).tobytes(), np.uint32)[0]) & 1)
        if best is None or key < best[0]:
            best = (key, float(cand))
    return best[1]


def exact_round_half_even(x: Fraction) -> int:
    f = x.numerator // x.denominator          # floor
    r = x - f
    if r > Fraction(1, 2):
        return f + 1
    if r < Fraction(1, 2):
        return f
    return f if f % 2 == 0 else f + 1


def brute_quantize(w):
    """Row by row from the definition, in exact rationals."""
    q = np.zeros(w.shape, np.int64)
    s = np.zeros(w.shape[0])
    for r in range(w.shape[0]):
        a = max(abs(Fraction(float(v))) for v in w[r])
        sr = exact_fp32_nearest(a / 127) if a else 0.0
        s[r] = sr
        for k in range(w.shape[1]):
            if sr == 0.0:
                continue
            q[r, k] = max(-127, min(127, exact_round_half_even(Fraction(float(w[r, k])) / Fraction(sr))))
    return q, s


def bf16_rows(rng, shape, std=0.02):
    return om.round_to_bf16(rng.normal(0, std, size=shape))


def test_quantize_matches_exact_rational_definition():
    rng = np.random.default_rng(3)
    w = bf16_rows(rng, (24, 96))
    w[5] = om.round_to_bf16(rng.normal(0, 7.0, 96))         # large values
    w[6] = om.round_to_bf16(rng.normal(0, 1e-6, 96))        # tiny values
    q, s = om.quantize_int8_rows(w)
    qb, sb = brute_quantize(w)
    np.testing.assert_array_equal(s.astype(np.float64), sb)
    np.testing.assert_array_equal(q.astype(np.int64), qb)


def test_quantize_ties_go_to_even():
    # s = fp32(127 / 127) = 1 exactly: w / s is w itself, and the half-integer
    # values must round to the even neighbour
    w = np.array([[127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, 100.5, -126.5]])
    q, s = om.quantize_int8_rows(w)
    assert s[0] == np.float32(1.0)
    np.testing.assert_array_equal(q[0], [127, 0, 2, 2, 0, -2, -2, 4, 100, -126])


def test_quantize_hand_worked_row():
    # a = 0.5; 0.5 / 127 = 0.0039370078740157...; the nearest fp32 is
    # 8454660 * 2^-31 = 0.00393700786, just below the real quotient, so the
    # scale is rounded before q is formed: 0.25 / s = 63.5000002 -> 64 (a
    # distance decision, not a tie), 0.125 / s = 31.7500001 -> 32,
    # 0.375 / s = 95.2500004 -> 95, and +-0.5 / s = 127.0000005 -> +-127
    w = np.array([[0.5, -0.25, 0.125, 0.0, -0.5, 0.375]])
    q, s = om.quantize_int8_rows(w)
    assert s[0] == np.float32(8454660 * 2.0 ** -31)
    assert float(s[0]) < 0.5 / 127
    np.testing.assert_array_equal(q[0], [127, -64, 32, 0, -127, 95])


def test_quantize_invariants():
    rng = np.random.default_rng(5)
    w = bf16_rows(rng, (16, 64))
    q, s = om.quantize_int8_rows(w)
    # the largest magnitude of every row maps to +-127
    idx = np.argmax(np.abs(w), axis=1)
    np.testing.assert_array_equal(np.abs(q[np.arange(16), idx]), 127)
    # sign symmetry
    qn, sn = om.quantize_int8_rows(-w)
    np.testing.assert_array_equal(qn, -q)
    np.testing.assert_array_equal(sn, s)
    # a power-of-two scale of a row scales s exactly and leaves q alone
    q4, s4 = om.quantize_int8_rows(w * 4.0)
    np.testing.assert_array_equal(q4, q)
    np.testing.assert_array_equal(s4, s * np.float32(4.0))
    # dequantisation error at most half a step
    err = np.abs(om.dequantize_int8_rows(q, s) - w)
    assert np.all(err <= s.astype(np.float64)[:, None] / 2 * (1 + 1e-12))
    # zero rows
    qz, sz = om.quantize_int8_rows(np.zeros((2, 8)))
    assert not qz.any() and not sz.any()


def small_weights(rng, cfg):
    d, hq, hkv, hd, F, V = cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim, cfg.vocab
    w = {"embed": bf16_rows(rng, (V, d), 1.0), "lm_head": bf16_rows(rng, (V, d), 0.3),
         "final_norm": np.ones(d)}
    for l in range(cfg.n_layers):
        w[f"{l}.attn_norm"] = np.ones(d)
        w[f"{l}.ffn_norm"] = np.ones(d)
        w[f"{l}.wq"] = bf16_rows(rng, (hq * hd, d), 0.3)
        w[f"{l}.wk"] = bf16_rows(rng, (hkv * hd, d), 0.3)
        w[f"{l}.wv"] = bf16_rows(rng, (hkv * hd, d), 0.3)
        w[f"{l}.wo"] = bf16_rows(rng, (d, hq * hd), 0.3)
        w[f"{l}.w_gate"] = bf16_rows(rng, (F, d), 0.3)
        w[f"{l}.w_up"] = bf16_rows(rng, (F, d), 0.3)
        w[f"{l}.w_down"] = bf16_rows(rng, (d, F), 0.3)
    return w


def test_int8_model_is_the_model_of_the_dequantised_weights():
    """weight_format="int8" runs the same decoder over q * s of every
    streamed matrix and leaves the embedding and the gains alone."""
    rng = np.random.default_rng(9)
    cfg = om.ModelConfig(2, 16, 2, 1, 8, 24, 32)
    w = small_weights(rng, cfg)
    deq = {}
    for k, v in w.items():
        if k.split(".")[-1] in om.INT8_MATRICES:
            deq[k] = om.dequantize_int8_rows(*om.quantize_int8_rows(v))
        else:
            deq[k] = v
    m8 = om.OracleModel(cfg, w, weight_format="int8")
    md = om.OracleModel(cfg, deq)
    mb = om.OracleModel(cfg, w)
    rows = [(0, 3, 0, 0), (0, 7, 1, 0), (0, 11, 2, 1), (1, 5, 0, 1)]
    z8 = om.step(m8, {0: om.SequenceKV(cfg, 8), 1: om.SequenceKV(cfg, 8)}, rows)
    zd = om.step(md, {0: om.SequenceKV(cfg, 8), 1: om.SequenceKV(cfg, 8)}, rows)
    zb = om.step(mb, {0: om.SequenceKV(cfg, 8), 1: om.SequenceKV(cfg, 8)}, rows)
    np.testing.assert_array_equal(z8, zd)
    assert np.abs(z8 - zb).max() > 1e-6          # quantisation does change the logits
    np.testing.assert_array_equal(m8.embed_rows([3]), mb.embed_rows([3]))


@pytest.mark.parametrize("mistake", ["per_column", "truncate", "no_clamp_scale"])
def test_planted_quantizer_mistakes_are_caught(mistake, monkeypatch):
    """Plausible slips in the quantiser fail the exact-rational pin."""
    real = om.quantize_int8_rows

    def bad(w):
        w = np.asarray(w, dtype=np.float64)
        if mistake == "per_column":
            a = np.max(np.abs(w), axis=0)
            s = (a.astype(np.float32) / np.float32(127.0)).astype(np.float32)
            q = np.clip(np.rint(w / s.astype(np.float64)[None, :]), -127, 127).astype(np.int8)
            return q, np.max(s) * np.ones(w.shape[0], np.float32)
        if mistake == "truncate":
            q, s = real(w)
            return np.clip(np.trunc(w / s.astype(np.float64)[:, None]), -127, 127).astype(np.int8), s
        a = np.max(np.abs(w), axis=1)
        s = (a / 127.0)                      # fp64 scale, not rounded to fp32
        return np.clip(np.rint(w / s[:, None]), -127, 127).astype(np.int8), s.astype(np.float32)

    monkeypatch.setattr(om, "quantize_int8_rows", bad)
    with pytest.raises(AssertionError):
        test_quantize_matches_exact_rational_definition()
