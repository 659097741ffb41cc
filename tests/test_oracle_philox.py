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


def test_draft_noise_group_word_fixes_each_groups_maximum():
    """What the group word must do, checked from its stated role rather than its formula: in
    every group of 16 entries, the largest variate sits at the position in the word's low four
    bits, equals the Gumbel variate of the word's uniform plus log 16 (the maximum of 16
    independent Gumbels is distributed so), and every other entry of the group is smaller.
    The word itself comes from the generator pinned to cuRAND above (stream 0, counter G >> 2)."""
    V, b, i = 16 * 96, 2, 5
    g = draft_gumbel(3, 4, np.array([b]), i, V)[0].reshape(-1, 16)
    for G in range(g.shape[0]):
        W = np.uint64(philox_words(3, 4, G >> 2, b, 0, i)[G & 3])
        p = int(W & np.uint64(15))
        assert int(np.argmax(g[G])) == p
        np.testing.assert_allclose(g[G, p], gumbel_from_word(W) + np.log(16.0), rtol=0, atol=1e-12)
        assert np.all(np.delete(g[G], p) < g[G, p])


def _noise(n_req=8, V=16 * 4096, seed=9, i=2):
    return draft_gumbel(seed, 1, np.arange(n_req), i, V)


def test_draft_noise_marginal_is_standard_gumbel():
    g = _noise().ravel()
    assert stats.kstest(g, stats.gumbel_r.cdf).pvalue > 0.01
    # every entry lies below the largest group variate: E_min >= -log(1 - 2^-24) / 16
    assert g.max() <= -np.log(-np.log(1.0 - 2.0 ** -24) / 16)


def test_draft_noise_group_maximum_is_gumbel_plus_log16_at_a_uniform_position():
    # the largest of 16 independent standard Gumbels is distributed as Gumbel + log 16, and
    # falls on each of the 16 positions with probability 1/16
    g = _noise().reshape(-1, 16)
    top = g.max(axis=1)
    assert stats.kstest(top - np.log(16.0), stats.gumbel_r.cdf).pvalue > 0.01
    counts = np.bincount(g.argmax(axis=1), minlength=16)
    assert stats.chisquare(counts).pvalue > 0.01
    # the smallest is distributed as the smallest of 16 Gumbels: P(min <= x) = 1 - (1 - F(x))^16
    low = g.min(axis=1)
    assert stats.kstest(low, lambda x: 1.0 - (1.0 - stats.gumbel_r.cdf(x)) ** 16).pvalue > 0.01


@pytest.mark.parametrize("k1,k2", [(0, 1), (3, 11), (0, 15), (15, 16)])
def test_draft_noise_entries_are_independent(k1, k2):
    # entries of one group, and the last entry of a group with the first of the next: the joint
    # law of (F(g1), F(g2)) is uniform on the unit square (F = standard Gumbel cdf)
    g = _noise(n_req=16)
    a = stats.gumbel_r.cdf(g[:, k1::32].ravel())
    b = stats.gumbel_r.cdf(g[:, k2::32].ravel())
    joint = np.histogram2d(a, b, bins=8, range=[[0, 1], [0, 1]])[0].ravel()
    assert stats.chisquare(joint).pvalue > 0.01
    assert abs(np.corrcoef(a, b)[0, 1]) < 0.01


def test_draft_noise_depends_on_request_step_and_offset():
    base = draft_gumbel(9, 1, np.array([4]), 2, 256)
    for other in (draft_gumbel(9, 1, np.array([5]), 2, 256), draft_gumbel(9, 1, np.array([4]), 3, 256),
                  draft_gumbel(9, 2, np.array([4]), 2, 256), draft_gumbel(10, 1, np.array([4]), 2, 256)):
        assert np.mean(base == other) < 0.01
    # a prefix of the vocabulary draws the same values
    np.testing.assert_array_equal(draft_gumbel(9, 1, np.array([4]), 2, 100), base[:, :100])
