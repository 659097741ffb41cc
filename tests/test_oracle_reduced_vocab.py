"""Pins of the reduced-vocabulary sampler: identity tables reduce to the plain sampler, the two
table conventions agree, and the law of the mapped token equals softmax over the scattered
target-size buffer (the page's construction, -inf off the draft positions)."""
import numpy as np
from scipy import stats

from oracle import markov_sample, map_to_target, markov_sample_reduced
from oracle.reduced_vocab import MODE_INDEX, MODE_OFFSET


def _inputs(seed, B=3, N=4, Vd=20, r=4):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, N, Vd)), rng.integers(0, Vd, B), rng.standard_normal((Vd, r)),
            rng.standard_normal((Vd, r)) * 0.3, np.full(B, 1.0))


def test_identity_tables_give_the_plain_sampler():
    L, a, w1, w2, T = _inputs(1)
    ref, _, _ = markov_sample(L, a, w1, w2, T, 5, 0)
    Vd = L.shape[2]
    t1, d1, _, _ = markov_sample_reduced(L, a, w1, w2, T, 5, 0, np.arange(Vd), MODE_INDEX, Vd)
    t2, d2, _, _ = markov_sample_reduced(L, a, w1, w2, T, 5, 0, np.zeros(Vd, np.int64), MODE_OFFSET, Vd)
    np.testing.assert_array_equal(t1, ref)
    np.testing.assert_array_equal(t2, ref)
    np.testing.assert_array_equal(d1, ref)


def test_index_and_offset_tables_agree_and_the_chain_stays_in_draft_ids():
    L, a, w1, w2, T = _inputs(2)
    Vd, Vt = L.shape[2], 500
    rng = np.random.default_rng(3)
    idx = np.sort(rng.choice(Vt, Vd, replace=False))
    t_i, d_i, _, _ = markov_sample_reduced(L, a, w1, w2, T, 7, 1, idx, MODE_INDEX, Vt)
    t_o, d_o, _, _ = markov_sample_reduced(L, a, w1, w2, T, 7, 1, idx - np.arange(Vd), MODE_OFFSET, Vt)
    np.testing.assert_array_equal(t_i, t_o)
    np.testing.assert_array_equal(t_i, idx[d_i])
    ref, _, _ = markov_sample(L, a, w1, w2, T, 7, 1)          # the chain itself does not see the table
    np.testing.assert_array_equal(d_i, ref)


def test_out_of_range_targets_are_minus_one():
    assert list(map_to_target(np.array([0, 1, 2]), np.array([5, 9, -1]), MODE_INDEX, 8)) == [5, -1, -1]
    assert list(map_to_target(np.array([0, 2]), np.array([7, 0, 6]), MODE_OFFSET, 8)) == [7, -1]


def test_law_of_the_mapped_token_is_softmax_over_the_scattered_buffer():
    """One step, many requests: the mapped first token follows softmax of the target-size buffer
    holding the draft logits at d2t positions and -inf elsewhere (chi-square, p > 1e-3)."""
    Vd, Vt, B = 6, 15, 60000
    rng = np.random.default_rng(9)
    base = rng.standard_normal(Vd)
    idx = np.array([13, 2, 7, 0, 11, 4])
    L = np.broadcast_to(base, (B, 1, Vd)).copy()
    t, _, _, _ = markov_sample_reduced(L, np.zeros(B, np.int64), np.zeros((Vd, 2)), np.zeros((Vd, 2)),
                                       np.ones(B), 21, 0, idx, MODE_INDEX, Vt)
    buf = np.full(Vt, -np.inf)
    buf[idx] = base
    p = np.exp(buf - buf.max())
    p /= p.sum()
    counts = np.bincount(t[:, 0], minlength=Vt)
    assert counts[p == 0].sum() == 0
    _, pval = stats.chisquare(counts[p > 0], B * p[p > 0])
    assert pval > 1e-3
