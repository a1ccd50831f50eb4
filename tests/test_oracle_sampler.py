"""Pins for the sampler oracle (CPU only): hand-worked examples, reductions
to greedy, the counter recurrence's closed form, and a chi-square test of the
draw against the softmax distribution."""
import math
import os

import numpy as np
import pytest

from oracle import philox
from oracle import sampler as os_

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(kind):
    out = []
    with open(os.path.join(GOLDEN, "sampler_examples.txt")) as f:
        for line in f:
            if line.startswith(kind + " "):
                out.append([float(v) for v in line.split()[1:]])
    return out


def P(**kw):
    base = dict(temperature=1.0, top_p=1.0, top_k=0, presence_penalty=0.0,
                frequency_penalty=0.0, penalty_decay=0.996)
    base.update(kw)
    return os_.SamplingParams(**base)


def test_penalty_examples():
    for l, c, pres, freq, want in golden("penalty"):
        got = os_.penalize(np.array([l]), np.array([c]), pres, freq)[0]
        assert got == np.float32(want)


def test_penalty_is_not_fused():
    """(l - f*c) with separate roundings differs from a fused multiply-add on
    a case chosen so the product is inexact in fp32."""
    l, c, f = np.float32(1.0), np.float32(1.0000001), np.float32(0.9999999)
    got = os_.penalize(np.array([l]), np.array([c]), 0.0, float(f))[0]
    sep = np.float32(l - np.float32(f * c))
    fused = np.float32(np.float64(l) - np.float64(f) * np.float64(c))
    assert got == sep
    assert sep != fused


def test_top_p_examples():
    logits = np.log(np.array([0.5, 0.3, 0.2])).astype(np.float32)
    for top_p, u, want in golden("topp"):
        tok = os_.sample_row(logits, np.zeros(3, np.float32), P(top_p=top_p), u)
        assert tok == int(want), (top_p, u)


def test_greedy_ties_to_lowest_id():
    l = np.array([0.5, 2.0, -1.0, 2.0], np.float32)
    assert os_.sample_row(l, np.zeros(4, np.float32), P(temperature=0.0), 0.9) == 1
    assert os_.sample_row(l, np.zeros(4, np.float32), P(top_k=1), 0.9) == 1


def test_top_k_ties_keep_lower_ids():
    l = np.array([1.0, 3.0, 3.0, 3.0, 0.0], np.float32)
    ids, pk, _ = os_.kept_set(l, P(top_k=2))
    assert list(ids) == [1, 2]
    np.testing.assert_allclose(pk, [0.5, 0.5])


def test_reductions_to_greedy():
    rng = np.random.default_rng(0)
    for _ in range(50):
        l = rng.normal(0, 2, 200).astype(np.float32)
        c = (rng.random(200) < 0.1).astype(np.float32) * rng.integers(1, 4, 200)
        g = os_.sample_row(l, c, P(temperature=0.0, frequency_penalty=1.0), 0.3)
        for u in (0.0, 0.5, 0.999999):
            assert os_.sample_row(l, c, P(top_k=1, frequency_penalty=1.0), u) == g
            assert os_.sample_row(l, c, P(top_p=1e-9, frequency_penalty=1.0), u) == g


def test_draw_frequencies_match_softmax():
    """T=1, top_p=1, top_k=0: frequencies of 40000 Philox-driven draws match
    softmax(logits) (chi-square, 15 dof)."""
    rng = np.random.default_rng(1)
    l = rng.normal(0, 1, 16).astype(np.float32)
    p = np.exp(l.astype(np.float64) - l.max())
    p /= p.sum()
    n = 40000
    counts = np.zeros(16)
    for i in range(n):
        u = philox.sampler_uniform(99, 7, i)
        counts[os_.sample_row(l, np.zeros(16, np.float32), P(), u)] += 1
    chi2 = np.sum((counts - n * p) ** 2 / (n * p))
    assert chi2 < 37.7          # p ~ 0.0015 upper tail for 15 dof


def test_temperature_scales_logits():
    """Logits a*l at temperature a*T keep the same distribution (a = 2 is exact)."""
    rng = np.random.default_rng(2)
    l = rng.normal(0, 1, 64).astype(np.float32)
    i1, p1, _ = os_.kept_set(l, P(temperature=0.7, top_p=0.8))
    i2, p2, _ = os_.kept_set((2 * l).astype(np.float32), P(temperature=1.4, top_p=0.8))
    np.testing.assert_array_equal(i1, i2)
    np.testing.assert_allclose(p1, p2, rtol=1e-12)


def test_counter_closed_form():
    for n, want in golden("counter"):
        c = np.zeros(4, np.float32)
        for _ in range(int(n)):
            c = os_.update_counters(c, 2, 0.996)
        assert abs(float(c[2]) - want) <= 1e-6 * want
    c = np.zeros(4, np.float32)
    for n in range(1, 2001):
        c = os_.update_counters(c, 1, 0.996)
        if n % 250 == 0:
            exact = (1 - 0.996 ** n) / 0.004
            assert abs(float(c[1]) - exact) <= 2e-4 * exact
    assert c[0] == 0 and c[3] == 0


def test_counter_decay_of_other_tokens():
    c = np.array([1.0, 0.0, 5.0], np.float32)
    c2 = os_.update_counters(c, 1, 0.996)
    assert c2[0] == np.float32(np.float32(1.0) * np.float32(0.996))
    assert c2[2] == np.float32(np.float32(5.0) * np.float32(0.996))
    assert c2[1] == np.float32(1.0)


# ---------------------------------------------------------------- forbidden tokens
def test_forbidden_greedy_takes_the_best_allowed():
    l = np.array([0.5, 3.0, 2.0, 2.5, -1.0], np.float32)
    c = np.zeros(5, np.float32)
    p = os_.SamplingParams(temperature=0.0, frequency_penalty=0.0)
    assert os_.sample_row(l, c, p, 0.5) == 1
    assert os_.sample_row(l, c, p, 0.5, forbidden=[1]) == 3
    assert os_.sample_row(l, c, p, 0.5, forbidden=[1, 3]) == 2
    assert os_.sample_row(l, c, p, 0.5, forbidden=[0, 1, 2, 3]) == 4     # the only allowed id


def test_forbidden_equals_removing_the_ids_from_the_vocabulary():
    """With ids removed, sampling over the rest (renumbered) is the same draw:
    the mask reduces to the unmasked algorithm on a smaller vocabulary."""
    rng = np.random.default_rng(3)
    for trial in range(200):
        V = 40
        l = rng.normal(0, 2, V).astype(np.float32)
        c = np.where(rng.random(V) < 0.2, rng.integers(1, 4, V), 0).astype(np.float32)
        bad = sorted(rng.choice(V, size=int(rng.integers(1, 12)), replace=False).tolist())
        keep = np.array([i for i in range(V) if i not in bad])
        p = os_.SamplingParams(temperature=float(rng.choice([0.0, 0.7, 1.0])), top_p=float(rng.choice([0.3, 0.9, 1.0])),
                             top_k=int(rng.choice([0, 5])), frequency_penalty=0.5, presence_penalty=0.25)
        u = float(rng.random())
        got = os_.sample_row(l, c, p, u, forbidden=bad)
        ref = int(keep[os_.sample_row(l[keep], c[keep], p, u)])
        assert got == ref and got not in bad


def test_forbidden_ids_are_never_drawn():
    rng = np.random.default_rng(4)
    l = np.zeros(16, np.float32)
    l[3] = 5.0                                     # would dominate the nucleus
    c = np.zeros(16, np.float32)
    p = os_.SamplingParams(temperature=1.0, top_p=1.0, frequency_penalty=0.0)
    seen = {os_.sample_row(l, c, p, float(rng.random()), forbidden=[3, 7]) for _ in range(500)}
    assert not seen & {3, 7} and len(seen) >= 12
