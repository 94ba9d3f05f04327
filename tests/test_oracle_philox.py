"""Pins of the oracle's Philox4x32-10 (CPU only).

The library pin is cuRAND's host-side Philox4_32_10 generator (runs on the CPU,
no GPU): its output block j for seed s is Philox4x32-10 of counter (0, 0, j, 0)
under key (s mod 2^32, s >> 32).  After the first round every state word is
non-zero, so a wrong multiplier, Weyl constant, word permutation or round count
changes the output.
"""

import ctypes

import numpy as np
import pytest

from oracle import philox as P


def _curand():
    for name in ("libcurand.so", "libcurand.so.10", "/usr/local/cuda/lib64/libcurand.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    pytest.skip("libcurand not loadable")


CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161


@pytest.mark.parametrize("seed", [0, 1234, 0x123456789ABCDEF0, (1 << 64) - 1])
def test_philox_matches_curand_host_generator(seed):
    lib = _curand()
    gen = ctypes.c_void_p()
    if lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) != 0:
        pytest.skip("curand host generator unavailable")
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        nblk = 50000
        out = np.zeros(4 * nblk, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(4 * nblk)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    ctr = np.zeros((nblk, 4), dtype=np.uint64)
    ctr[:, 2] = np.arange(nblk)
    ref = P.philox4x32(ctr, P.seed_key(seed))
    assert np.array_equal(ref, out.reshape(nblk, 4))


def test_sr_bits_layout():
    # element i takes counter i//8, word (i//2)%4, low half for even i, high half for odd i
    seed = 99
    idx = np.arange(64, dtype=np.uint64)
    r = P.sr_bits16(seed, idx)
    ctr = np.zeros((8, 4), dtype=np.uint64)
    ctr[:, 0] = np.arange(8)
    blocks = P.philox4x32(ctr, P.seed_key(seed))
    for i in range(64):
        w = int(blocks[i // 8][(i // 2) % 4])
        assert r[i] == ((w >> (16 * (i % 2))) & 0xFFFF)
    # high counter word carries index // 8 >> 32
    big = np.array([(1 << 35) * 8 + 3], dtype=np.uint64)
    c = np.array([[0, 1 << 3, 0, 0]], dtype=np.uint64)
    w = P.philox4x32(c, P.seed_key(seed))[0][1]
    assert P.sr_bits16(seed, big)[0] == (w >> 16) & 0xFFFF


def test_sr_bits_uniform_chi2():
    r = P.sr_bits16(5, np.arange(1 << 20, dtype=np.uint64))
    assert r.max() < 65536
    hist = np.bincount((r >> 8).astype(np.int64), minlength=256)
    exp = len(r) / 256
    chi2 = float(((hist - exp) ** 2 / exp).sum())
    # 255 dof: mean 255, sd ~22.6; 6 sd band
    assert 120 < chi2 < 400, chi2
