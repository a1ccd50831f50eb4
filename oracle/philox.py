"""Philox-4x32-10 counter-based generator (oracle copy).

TEST INFRASTRUCTURE ONLY -- see the package docstring for who may import it.

Definition: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
1, 2, 3", SC'11, section on the Philox family.  State is a 4-word counter
(c0, c1, c2, c3) and a 2-word key (k0, k1), all 32-bit.  One round with
multipliers M0 = 0xD2511F53, M1 = 0xCD9E8D57:

    hi0:lo0 = M0 * c0 (64-bit product),  hi1:lo1 = M1 * c2
    (c0, c1, c2, c3) <- (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0)

and between rounds the key is bumped by the Weyl constants
(W0, W1) = (0x9E3779B9, 0xBB67AE85).  Ten rounds give Philox-4x32-10.

How the sampler uses it (a reading, listed in the design notes): the key is
(seed mod 2^32, seed >> 32), the counter is (token_index, request_id mod 2^32,
request_id >> 32, 0) and the uniform is (out0 >> 8) * 2^-24, in [0, 1).
Keying by request rather than slot keeps draws independent of placement.

Pinning: the round structure above is checked against cuRAND's host
Philox-4x32-10 generator (an independent implementation of the same
published definition) in the CPU tests when libcurand is available; without
it this module is parity unpinned and only statistical checks run.
"""
from __future__ import annotations

import numpy as np

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
MASK = 0xFFFFFFFF


def philox4x32_10(counter, key):
    """Vectorised over leading axes: counter [..., 4], key [..., 2] (uint32)."""
    c = np.asarray(counter, dtype=np.uint64) & MASK
    k = np.asarray(key, dtype=np.uint64) & MASK
    c0, c1, c2, c3 = (c[..., i].copy() for i in range(4))
    k0, k1 = k[..., 0].copy(), k[..., 1].copy()
    for r in range(10):
        if r:
            k0 = (k0 + W0) & MASK
            k1 = (k1 + W1) & MASK
        p0 = c0 * np.uint64(M0)          # < 2^64: exact in uint64
        p1 = c2 * np.uint64(M1)
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def sampler_uniform(seed: int, request_id: int, token_index: int) -> float:
    """The sampler's uniform for one (request, generated-token index)."""
    ctr = [token_index & MASK, request_id & MASK, (request_id >> 32) & MASK, 0]
    key = [seed & MASK, (seed >> 32) & MASK]
    out0 = int(philox4x32_10(ctr, key)[0])
    return (out0 >> 8) * (2.0 ** -24)
