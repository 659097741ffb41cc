"""Pins for the oracle's Philox4x32-10 and its uniform / Gumbel variates.

The generator is pinned against an independent implementation: cuRAND's
host-side PHILOX4_32_10 generator (a library routine that runs on the CPU).
Observed layout of that generator: output n for seed s is word n mod 4 of
block m = floor(n / 4), and block m is the Philox output of counter
(floor(m / 65536), 0, m mod 65536, 0) under key (lo32(s), hi32(s)); the
generator offset adds to n, so a large offset carries into the second word.
This pins the round function, the key schedule and the counter words c0, c1
and c2.  The fourth word c3 is exercised only through the symmetric round
structure and the GPU/oracle agreement of independent implementations.
"""
import ctypes
import ctypes.util
import glob
import os

import numpy as np
import pytest
from scipy import stats

from oracle.philox import (philox4x32_10, philox_words, uniform_from_word,
                           gumbel_from_word, draft_gumbel)

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _curand():
    cands = []
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cands += sorted(glob.glob(os.path.join(home, "lib64", "libcurand.so*")))
    cands += sorted(glob.glob(os.path.join(home, "targets", "*", "lib", "libcurand.so*")))
    lib = ctypes.util.find_library("curand")
    if lib:
        cands.append(lib)
    for c in cands:
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    pytest.skip("libcurand not found")


def _curand_words(seed: int, count: int, offset: int = 0) -> np.ndarray:
    cr = _curand()
    gen = ctypes.c_void_p()
    CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161
    st = cr.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10)
    if st != 0:
        pytest.skip(f"curandCreateGeneratorHost failed ({st})")
    try:
        assert cr.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert cr.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        out = np.zeros(count, dtype=np.uint32)
        st = cr.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(count))
        assert st == 0, st
    finally:
        cr.curandDestroyGenerator(gen)
    return out


@pytest.mark.parametrize("seed", [0, 1, 0xDEADBEEF, 0x0123456789ABCDEF, 2 ** 64 - 1])
def test_philox_matches_curand_host_generator(seed):
    n_blk = 65536 + 4096
    ref = _curand_words(seed, 4 * n_blk).reshape(n_blk, 4)
    m = np.arange(n_blk, dtype=np.uint64)
    w = philox4x32_10(m >> np.uint64(16), 0, m & np.uint64(0xFFFF), 0,
                      seed & 0xFFFFFFFF, seed >> 32)
    got = np.stack(w, axis=1).astype(np.uint32)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("c1", [1, 7, 0x3FFE])   # the 64-bit offset limits c1 to 14 bits
def test_philox_second_counter_word_matches_curand(c1):
    # block m = ((c1 << 32) + c0) * 65536 + c2 is counter (c0, c1, c2, 0)
    c0 = 0xFFFFFFFF
    seed = 0x5EED
    m0 = ((c1 << 32) + c0) * 65536 + 65536 - 32        # 32 blocks before a carry into c1
    ref = _curand_words(seed, 4 * 64, offset=4 * m0).reshape(64, 4)
    m = [m0 + t for t in range(64)]
    hi = np.array([x >> 16 for x in m], dtype=np.uint64)
    c0s = hi & np.uint64(0xFFFFFFFF)
    c1s = hi >> np.uint64(32)
    c2s = np.array([x & 0xFFFF for x in m], dtype=np.uint64)
    got = np.stack(philox4x32_10(c0s, c1s, c2s, 0, seed, 0), axis=1).astype(np.uint32)
    np.testing.assert_array_equal(got, ref)


def test_counter_layout_words():
    # philox_words places (j, b, stream<<16 | i, offset) into the four counter words
    seed, off = 0xABCDEF0123456789, 77
    a = philox_words(seed, off, 5, 3, 2, 9)
    b = philox4x32_10(5, 3, (2 << 16) | 9, 77, seed & 0xFFFFFFFF, seed >> 32)
    assert all(int(x) == int(y) for x, y in zip(a, b))
    # all four words differ between neighbouring counters in every position
    base = np.array(philox4x32_10(0, 0, 0, 0, 1, 2))
    for pos in range(4):
        c = [0, 0, 0, 0]
        c[pos] = 1
        other = np.array(philox4x32_10(*c, 1, 2))
        assert np.all(base != other)


def test_uniform_is_exact_float32_in_open_interval():
    w = np.array([0, 1, 511, 512, 2 ** 31, 2 ** 32 - 1], dtype=np.uint64)
    u = uniform_from_word(w)
    assert u.min() == 2.0 ** -24 and u.max() == 1.0 - 2.0 ** -24
    assert np.all(u.astype(np.float32).astype(np.float64) == u)     # exactly representable
    assert np.all((u > 0) & (u < 1))


def test_uniform_chi_square():
    words = philox4x32_10(np.arange(250_000, dtype=np.uint64), 11, 22, 33, 44, 55)
    u = uniform_from_word(np.concatenate(words))
    counts, _ = np.histogram(u, bins=256, range=(0.0, 1.0))
    p = stats.chisquare(counts).pvalue
    assert p > 0.01, p


def test_gumbel_distribution_and_bounds():
    g = gumbel_from_word(np.concatenate(philox4x32_10(np.arange(250_000, dtype=np.uint64), 1, 2, 3, 4, 5)))
    # Kolmogorov-Smirnov against the standard Gumbel law (scipy's gumbel_r)
    assert stats.kstest(g, stats.gumbel_r.cdf).pvalue > 0.01
    # support of the discretised variate: u in [2^-24, 1-2^-24]
    gmax = -np.log(-np.log(1.0 - 2.0 ** -24))
    gmin = -np.log(-np.log(2.0 ** -24))
    assert g.max() <= gmax and g.min() >= gmin
    assert 16.63 < gmax < 16.64 and -2.82 < gmin < -2.81


def test_draft_gumbel_word_layout():
    # element v: high half from stream 0 and low half from stream 3, both from counter
    # v >> 3, word (v & 7) >> 1, bits 0-15 (even v) or 16-31 (odd v)
    g = draft_gumbel(3, 4, np.array([2]), 5, 20)
    for v in range(20):
        hw = philox_words(3, 4, v >> 3, 2, 0, 5)[(v & 7) >> 1]
        lw = philox_words(3, 4, v >> 3, 2, 3, 5)[(v & 7) >> 1]
        sh = 16 * (v & 1)
        word = (((int(hw) >> sh) & 0xFFFF) << 16) | ((int(lw) >> sh) & 0xFFFF)
        assert g[0, v] == gumbel_from_word(np.uint64(word))


def test_draft_words_uniform_and_halves_independent():
    from oracle.philox import draft_word, draft_halfword
    v = np.arange(200_000, dtype=np.uint64)
    w = draft_word(9, 1, 4, 2, v)
    counts, _ = np.histogram((w >> np.uint64(16)).astype(np.float64), bins=64, range=(0, 65536))
    assert stats.chisquare(counts).pvalue > 0.01
    counts, _ = np.histogram((w & np.uint64(0xFFFF)).astype(np.float64), bins=64, range=(0, 65536))
    assert stats.chisquare(counts).pvalue > 0.01
    hi = draft_halfword(9, 1, 4, 2, v, 0)
    lo = draft_halfword(9, 1, 4, 2, v, 3)
    joint = np.histogram2d((hi >> np.uint64(13)).astype(float), (lo >> np.uint64(13)).astype(float),
                           bins=8, range=[[0, 8], [0, 8]])[0].ravel()
    assert stats.chisquare(joint).pvalue > 0.01
    # neighbouring elements get different words (no sharing of halves)
    assert len(np.unique(w[:4096])) == 4096
