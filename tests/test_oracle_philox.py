"""Pins for the oracle's Philox4x32-10 and its threshold mapping.

The generator is defined in Salmon et al., "Parallel random numbers: as easy
as 1, 2, 3" (SC'11), which the S3R paper cites for its counter-based PRNG
(§II "The cost of randomness").  Pinned against a library routine: cuRAND's
host-side PHILOX4_32_10 generator, which runs on the CPU.  Its output stream
for seed s is  out[4*(j*65536 + i) + w] = Philox((j, 0, i, 0), (s_lo, s_hi))[w]
(64 Ki interleaved subsequences), checked at 46 counters per seed over a
2^22-word stream; counter words 0 and 2 and both key words vary there.
"""
import ctypes as C
import ctypes.util
import os

import numpy as np
import pytest


def _curand():
    cands = ["/usr/local/cuda/lib64/libcurand.so", "/usr/local/cuda/targets/sbsa-linux/lib/libcurand.so",
             "/usr/local/cuda/targets/x86_64-linux/lib/libcurand.so", ctypes.util.find_library("curand")]
    for c in cands:
        if not c:
            continue
        try:
            return C.CDLL(c)
        except OSError:
            continue
    pytest.skip("libcurand not available")


CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161


def curand_host_stream(seed: int, n: int) -> np.ndarray:
    L = _curand()
    g = C.c_void_p()
    assert L.curandCreateGeneratorHost(C.byref(g), C.c_int(CURAND_RNG_PSEUDO_PHILOX4_32_10)) == 0
    try:
        assert L.curandSetPseudoRandomGeneratorSeed(g, C.c_ulonglong(seed)) == 0
        out = np.zeros(n, dtype=np.uint32)
        assert L.curandGenerate(g, C.c_void_p(out.ctypes.data), C.c_size_t(n)) == 0
        return out
    finally:
        L.curandDestroyGenerator(g)


@pytest.mark.parametrize("seed", [0x1234567890ABCDEF, 0, 0xFFFFFFFF00000001, (77 << 32) | 5])
def test_philox_matches_curand_host_stream(orc, seed):
    n = 1 << 22
    stream = curand_host_stream(seed, n)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    subseqs = 65536
    rng = np.random.default_rng(seed & 0xFFFF)
    picks = [(0, 0), (0, 1), (0, 65535), (1, 0), (3, 17), (15, 65535)]
    picks += [(int(rng.integers(0, n // 4 // subseqs)), int(rng.integers(0, subseqs))) for _ in range(40)]
    for j, i in picks:
        base = 4 * (j * subseqs + i)
        got = orc.philox4x32_10([j, 0, i, 0], key)
        assert np.array_equal(got, stream[base:base + 4]), (j, i)


def test_token_threshold_is_curand_word(orc):
    """u_t = top 24 bits of word 0 of Philox(counter=(t,0,0,0), key=(seed, tensor_id))."""
    seed, tid = 0x0000BEEF, 7
    stream = curand_host_stream((tid << 32) | seed, 1 << 22)
    for t in [0, 1, 2, 5, 15]:
        w = int(stream[4 * (t * 65536 + 0)])
        assert orc.token_threshold(t, seed, tid) == (w >> 8) / 2.0 ** 24


def test_element_threshold_is_curand_word(orc):
    seed, tid = 3, 0x101
    stream = curand_host_stream((tid << 32) | seed, 1 << 22)
    for e in [0, 1, 2, 3, 4, 7, 33, 63]:
        c, w = e >> 2, e & 3
        word = int(stream[4 * (c * 65536) + w])
        assert orc.element_threshold(e, seed, tid) == (word >> 8) / 2.0 ** 24


def test_word_to_unit_grid(orc):
    assert orc.word_to_unit(0) == 0.0
    assert orc.word_to_unit(0xFF) == 0.0
    assert orc.word_to_unit(0x100) == 2.0 ** -24
    assert orc.word_to_unit(0xFFFFFFFF) == 1.0 - 2.0 ** -24


def test_token_thresholds_uniform_chi2(orc):
    """Chi-square test of u_t over 65536 tokens in 64 bins (df = 63)."""
    n, bins = 65536, 64
    u = np.array([orc.token_threshold(t, 0, 0) for t in range(n)])
    hist = np.bincount(np.minimum((u * bins).astype(int), bins - 1), minlength=bins)
    chi2 = float(((hist - n / bins) ** 2 / (n / bins)).sum())
    # df = 63: mean 63, sd ~ 11.2; reject only far tails
    assert 25 < chi2 < 120, chi2


def test_philox_avalanche(orc):
    """Flipping one input bit flips about half of the 128 output bits."""
    rng = np.random.default_rng(5)
    flips = []
    for _ in range(200):
        ctr = rng.integers(0, 2 ** 32, 4, dtype=np.uint64).astype(np.uint32)
        key = rng.integers(0, 2 ** 32, 2, dtype=np.uint64).astype(np.uint32)
        base = orc.philox4x32_10(ctr, key)
        which = int(rng.integers(0, 6))
        bit = np.uint32(1 << int(rng.integers(0, 32)))
        c2, k2 = ctr.copy(), key.copy()
        if which < 4:
            c2[which] ^= bit
        else:
            k2[which - 4] ^= bit
        out = orc.philox4x32_10(c2, k2)
        flips.append(sum(bin(int(a ^ b)).count("1") for a, b in zip(base, out)))
    m = np.mean(flips)
    assert abs(m - 64) < 3, m
