"""Philox4x32-10 counter-based generator (oracle; test infrastructure only).

The pages ask for stochastic rounding from a seeded generator but name none
(gonzo_ML #3986, section "Стохастическая квантизация"); the generator fixed
for this implementation is Philox4x32 with 10 rounds, written from its
published definition: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3", SC'11.

One round maps a counter (c0, c1, c2, c3) under a key (k0, k1) to

    (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0))

with the 32x32->64-bit products split into high and low halves; between
rounds the key is advanced by the Weyl constants (W0, W1).  All arithmetic is
modulo 2^32.

Stream layout used by the quantizer (one fixed reading): key = (seed & 0xffffffff,
seed >> 32).  Output element with linear index i (row-major in the OUTPUT
layout) takes counter (i // 8 low 32 bits, i // 8 high 32 bits, 0, 0), word
(i // 2) % 4 of the result, and from it the low 16 bits when i is even, the
high 16 bits when i is odd.  One generator call thus serves 8 elements.
"""

from __future__ import annotations

import numpy as np

PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint64(0x9E3779B9)
PHILOX_W1 = np.uint64(0xBB67AE85)
MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32(counter: np.ndarray, key: tuple, rounds: int = 10) -> np.ndarray:
    """Philox4x32-`rounds` of an array of counters.

    counter: uint32-valued array of shape (..., 4).  key: (k0, k1) Python ints.
    Returns a uint32 array of the same shape.
    """
    c = np.asarray(counter, dtype=np.uint64) & MASK32
    c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
    k0 = np.uint64(key[0] & 0xFFFFFFFF)
    k1 = np.uint64(key[1] & 0xFFFFFFFF)
    for r in range(rounds):
        if r > 0:
            k0 = (k0 + PHILOX_W0) & MASK32
            k1 = (k1 + PHILOX_W1) & MASK32
        p0 = PHILOX_M0 * c0  # < 2^64: exact in uint64
        p1 = PHILOX_M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def seed_key(seed: int) -> tuple:
    seed &= (1 << 64) - 1
    return (seed & 0xFFFFFFFF, seed >> 32)


def sr_bits16(seed: int, index: np.ndarray) -> np.ndarray:
    """16 random bits for each output-layout linear index (uint32 array < 2^16)."""
    index = np.asarray(index, dtype=np.uint64)
    block = index >> np.uint64(3)
    ctr = np.zeros(index.shape + (4,), dtype=np.uint64)
    ctr[..., 0] = block & MASK32
    ctr[..., 1] = block >> np.uint64(32)
    out = philox4x32(ctr, seed_key(seed))
    word = ((index >> np.uint64(1)) & np.uint64(3)).astype(np.int64)
    w = np.take_along_axis(out, word[..., None], axis=-1)[..., 0].astype(np.uint32)
    shift = ((index & np.uint64(1)) * np.uint64(16)).astype(np.uint32)
    return (w >> shift) & np.uint32(0xFFFF)
