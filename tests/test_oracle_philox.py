"""Pins for the Philox-4x32-10 oracle.

cuRAND ships an independent host implementation of Philox-4x32-10.  Its host
generator, seeded with s at offset 0, emits group g of four words from key
(s mod 2^32, s >> 32) and counter (g >> 16, 0, g mod 2^16, 0); an offset of
4*2^16*(2^32 + k) moves the first word's counter to k with a carry of one
into the second word.  Matching it pins the multipliers, the key schedule,
the round count and the output order.  Skipped where libcurand is absent.
"""
import ctypes
import ctypes.util
import glob

import numpy as np
import pytest

from oracle import philox


def _curand():
    cands = glob.glob("/usr/local/cuda/lib64/libcurand.so*") + [ctypes.util.find_library("curand") or ""]
    for c in cands:
        if c:
            try:
                return ctypes.CDLL(c)
            except OSError:
                pass
    return None


def curand_words(seed, offset, n):
    lib = _curand()
    if lib is None:
        pytest.skip("libcurand not available")
    gen = ctypes.c_void_p()
    if lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) != 0:   # PHILOX4_32_10
        pytest.skip("cuRAND host generator unavailable")
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        buf = (ctypes.c_uint * n)()
        assert lib.curandGenerate(gen, buf, ctypes.c_size_t(n)) == 0
        return np.frombuffer(buf, dtype=np.uint32).copy()
    finally:
        lib.curandDestroyGenerator(gen)


@pytest.mark.parametrize("seed", [0, 0x0123456789ABCDEF, 2 ** 64 - 1])
def test_matches_curand_host_generator(seed):
    n_groups = 1 << 17
    got = curand_words(seed, 0, 4 * n_groups).reshape(-1, 4)
    g = np.arange(n_groups, dtype=np.uint64)
    ctr = np.stack([g >> 16, 0 * g, g & 0xFFFF, 0 * g], -1)
    key = np.broadcast_to(np.array([seed & 0xFFFFFFFF, seed >> 32], dtype=np.uint64), (n_groups, 2))
    np.testing.assert_array_equal(philox.philox4x32_10(ctr, key), got)


def test_matches_curand_with_carry_into_second_word():
    seed, k = 0xDEADBEEFCAFEF00D, 5
    got = curand_words(seed, 4 * (1 << 16) * ((1 << 32) + k), 4 * 8).reshape(-1, 4)
    ctr = np.array([[k, 1, j, 0] for j in range(8)], dtype=np.uint64)
    key = np.array([[seed & 0xFFFFFFFF, seed >> 32]] * 8, dtype=np.uint64)
    np.testing.assert_array_equal(philox.philox4x32_10(ctr, key), got)


def test_sampler_uniform_range_and_uniformity():
    us = np.array([philox.sampler_uniform(12345, 3, i) for i in range(20000)])
    assert us.min() >= 0.0 and us.max() < 1.0
    assert np.all(us * 2 ** 24 == np.floor(us * 2 ** 24))      # 24-bit grid
    counts, _ = np.histogram(us, bins=20, range=(0, 1))
    chi2 = np.sum((counts - 1000) ** 2 / 1000)
    assert chi2 < 43.8         # 19 dof, upper tail ~ 0.001


def test_uniform_depends_on_request_not_slot():
    a = philox.sampler_uniform(1, 2 ** 40 + 3, 17)
    b = philox.sampler_uniform(1, 2 ** 40 + 4, 17)
    c = philox.sampler_uniform(1, 3, 17)
    assert len({a, b, c}) == 3
