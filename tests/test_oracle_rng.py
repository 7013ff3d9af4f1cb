"""Pins for the oracle's random streams (Philox4x32-10, uniform map, Gumbel).

The Philox bijection is compared with an independent implementation: the
cuRAND host-side PHILOX4_32_10 generator, which emits, for seed s, the blocks
philox(counter = (i mod 2^32, i >> 32, sub, 0), key = (s mod 2^32, s >> 32))
with 65536 interleaved subsequences ``sub``.  The uniform map and the Gumbel
transform are pinned by their lattice, their range and their moments.
"""
import ctypes
import ctypes.util
import math
import os

import numpy as np
import pytest

import oracle

CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161
SUBSEQ = 65536


def _curand():
    for path in ("/usr/local/cuda/lib64/libcurand.so", ctypes.util.find_library("curand")):
        if path and os.path.exists(path) if path.startswith("/") else path:
            try:
                return ctypes.CDLL(path)
            except OSError:
                continue
    return None


def _curand_words(seed, offset, n):
    lib = _curand()
    if lib is None:
        pytest.skip("libcurand not available")
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) == 0
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        out = np.zeros(n, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    return out


def test_philox_matches_curand_host_generator():
    seed = 1234567
    words = _curand_words(seed, 0, 4 * SUBSEQ * 2).reshape(2, SUBSEQ, 4)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    rng = np.random.default_rng(1)
    subs = list(range(4)) + list(rng.integers(0, SUBSEQ, 60))
    for i in range(2):
        for s in subs:
            got = oracle.philox4x32_10([i, 0, s, 0], key)
            np.testing.assert_array_equal(got, words[i, s], err_msg="counter %d sub %d" % (i, s))


def test_philox_high_counter_word_and_high_key_word():
    seed = (7 << 32) | 99
    i = (1 << 32) + 5  # counter word 0 = 5, word 1 = 1
    words = _curand_words(seed, 4 * SUBSEQ * i, 8).reshape(2, 4)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    np.testing.assert_array_equal(oracle.philox4x32_10([5, 1, 0, 0], key), words[0])
    np.testing.assert_array_equal(oracle.philox4x32_10([5, 1, 1, 0], key), words[1])


def test_philox_every_counter_word_changes_output():
    base = oracle.philox4x32_10([3, 4, 5, 6], [7, 8])
    for w in range(4):
        c = [3, 4, 5, 6]
        c[w] ^= 1
        assert not np.array_equal(oracle.philox4x32_10(c, [7, 8]), base)


def test_stream_layout_selects_word_by_token():
    # token v uses counter (v >> 2, j, request, stream) and word v & 3
    seed, rid, j, stream = (5 << 32) | 11, 77, 3, 2
    for v in (0, 1, 2, 3, 4, 9, 4095, 129279):
        blk = oracle.philox4x32_10([v >> 2, j, rid, stream], [seed & 0xFFFFFFFF, seed >> 32])
        assert oracle.random_word(seed, rid, j, v, stream) == int(blk[v & 3])


def test_uniform_lattice_and_range():
    u = oracle.uniforms(0, 5, 1, 0, 200000, 0)
    k2 = u * 2.0 ** 24
    assert np.all(k2 == np.round(k2)) and np.all(np.round(k2) % 2 == 1)
    assert u.min() > 0.0 and u.max() < 1.0
    assert np.all(u.astype(np.float32).astype(np.float64) == u)  # exact in fp32
    gmin = -math.log(-math.log(2.0 ** -24))
    gmax = -math.log(-math.log(1.0 - 2.0 ** -24))
    assert abs(gmin - (-2.8116)) < 1e-4 and abs(gmax - 16.6355) < 1e-4
    g = -np.log(-np.log(u))
    assert g.min() >= gmin and g.max() <= gmax


def test_uniform_chi_square_and_stream_independence():
    n = 1 << 20
    u = oracle.uniforms(42, 9, 0, 0, n, 1)
    counts = np.bincount((u * 256).astype(int), minlength=256)
    chi2 = ((counts - n / 256) ** 2 / (n / 256)).sum()
    # 255 degrees of freedom: mean 255, sd ~22.6; 6 sd bound
    assert chi2 < 255 + 6 * math.sqrt(2 * 255), chi2
    v = oracle.uniforms(42, 9, 0, 0, n, 2)
    corr = np.corrcoef(u, v)[0, 1]
    assert abs(corr) < 6 / math.sqrt(n)
    w = oracle.uniforms(42, 10, 0, 0, n, 1)
    assert abs(np.corrcoef(u, w)[0, 1]) < 6 / math.sqrt(n)


def test_gumbel_moments():
    n = 1 << 20
    u = oracle.uniforms(3, 1, 2, 0, n, 0)
    g = -np.log(-np.log(u))
    euler_gamma = 0.5772156649015329
    var = math.pi ** 2 / 6
    assert abs(g.mean() - euler_gamma) < 6 * math.sqrt(var / n)
    assert abs(g.var() - var) < 0.02
    assert oracle.gumbel(3, 1, 2, 17, 0) == pytest.approx(g[17], rel=0, abs=0)
