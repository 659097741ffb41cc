"""Pins of verification from logits (oracle side).

The rule is lossless, so whatever the draft, the emitted tokens follow the target: the
first emitted token follows target row 0, and given that the first draft token was
accepted the second follows target row 1 -- which holds only if the draft distribution
used at position 1 is the one conditioned on the right previous token.  Further pins:
the acceptance rate of position 0 equals 1 - TV(p_t, p_d), a greedy draft is accepted
with probability p_t(x), draft_lse reduces to scipy's logsumexp without a Markov bias,
and the Gumbel words are the Philox words of their counters."""
import numpy as np
import pytest
from scipy import stats
from scipy.special import logsumexp

from oracle import (verify_from_logits, draft_distributions, draft_lse, residual_gumbel,
                    markov_sample, philox4x32_10)


def _case(seed, V=6, r=3, gamma=2, bias_scale=1.5):
    rng = np.random.default_rng(seed)
    t = rng.standard_normal((gamma + 1, V)) * 1.5
    L = rng.standard_normal((gamma, V))
    w1 = rng.standard_normal((V, r))
    w2 = rng.standard_normal((V, r)) * bias_scale
    anchor = int(rng.integers(0, V))
    return t, L, w1, w2, anchor


def _batch(t, L, anchor, B):
    return (np.broadcast_to(t, (B,) + t.shape).copy(), np.broadcast_to(L, (B,) + L.shape).copy(),
            np.full(B, anchor))


def _target_law(row, T):
    return np.exp(row / T - logsumexp(row / T))


def _chi2_ok(samples, p, V):
    counts = np.bincount(samples, minlength=V)
    keep = p * len(samples) > 5
    exp = p[keep] * len(samples)
    obs = counts[keep]
    other = len(samples) - obs.sum()
    if (~keep).any():
        obs = np.append(obs, other)
        exp = np.append(exp, len(samples) - exp.sum())
    return stats.chisquare(obs, exp)[1]


@pytest.mark.parametrize("T_d", [1.3, 0.0])
def test_emitted_tokens_follow_the_target(T_d):
    B, V = 30000, 6
    t, L, w1, w2, a = _case(1, bias_scale=1.5 if T_d > 0 else 0.3)
    if T_d == 0:
        L = t[:2] / 0.8           # a greedy draft close to the target: its argmax is often accepted
    tb, Lb, anchor = _batch(t, L, a, B)
    Tt, Td = np.full(B, 0.8), np.full(B, T_d)
    x, _, _ = markov_sample(Lb, anchor, w1, w2, Td, 4, 0)
    out, nacc, _, _ = verify_from_logits(tb, Tt, Lb, anchor, w1, w2, Td, x, None, 5, 0)
    assert _chi2_ok(out[:, 0], _target_law(t[0], 0.8), V) > 1e-3
    sel = nacc >= 1
    assert 0.05 < sel.mean() < 0.95                       # a real mixture of accepts and rejects
    assert _chi2_ok(out[sel, 1], _target_law(t[1], 0.8), V) > 1e-3


def test_wrong_previous_token_would_be_detected(monkeypatch):
    """Planted mistake: the oracle's draft distribution at every position conditioned on the
    anchor instead of x_{k-1}.  The second emitted token is then biased, and the law test
    above rejects it."""
    import oracle.verify_logits as vl
    B, V = 30000, 6
    t, L, w1, w2, a = _case(1)
    tb, Lb, anchor = _batch(t, L, a, B)
    Tt, Td = np.full(B, 0.8), np.full(B, 1.3)
    x, _, _ = markov_sample(Lb, anchor, w1, w2, Td, 4, 0)
    monkeypatch.setattr(vl, "_prev_tokens",
                        lambda anc, toks: np.repeat(np.asarray(anc).reshape(-1, 1), np.shape(toks)[1], 1))
    out, nacc, _, _ = vl.verify_from_logits(tb, Tt, Lb, anchor, w1, w2, Td, x, None, 5, 0)
    sel = nacc >= 1
    assert _chi2_ok(out[sel, 1], _target_law(t[1], 0.8), V) < 1e-6


def test_acceptance_rate_of_position_zero_is_one_minus_tv():
    B, V = 40000, 6
    t, L, w1, w2, a = _case(2)
    tb, Lb, anchor = _batch(t, L, a, B)
    Tt, Td = np.full(B, 1.0), np.full(B, 0.7)
    x, _, _ = markov_sample(Lb, anchor, w1, w2, Td, 6, 0)
    _, nacc, _, _ = verify_from_logits(tb, Tt, Lb, anchor, w1, w2, Td, x, None, 7, 0)
    pt = _target_law(t[0], 1.0)
    pd = draft_distributions(Lb[:1], anchor[:1], w1, w2, Td[:1], x[:1])[0, 0]
    expect = 1.0 - 0.5 * np.abs(pt - pd).sum()
    rate = (nacc >= 1).mean()
    assert abs(rate - expect) < 5 * np.sqrt(expect * (1 - expect) / B)


def test_greedy_draft_is_accepted_with_the_target_probability():
    B, V = 40000, 6
    t, L, w1, w2, a = _case(3)
    tb, Lb, anchor = _batch(t, L, a, B)
    Td = np.zeros(B)
    x, _, _ = markov_sample(Lb, anchor, w1, w2, Td, 0, 0)
    _, nacc, _, _ = verify_from_logits(tb, np.ones(B), Lb, anchor, w1, w2, Td, x, None, 9, 0)
    p = _target_law(t[0], 1.0)[x[0, 0]]
    rate = (nacc >= 1).mean()
    assert abs(rate - p) < 5 * np.sqrt(p * (1 - p) / B)


def test_draft_lse_without_bias_is_logsumexp():
    rng = np.random.default_rng(4)
    B, g, V, r = 3, 4, 50, 5
    L = rng.standard_normal((B, g, V)) * 2
    w1 = np.zeros((V, r))
    w2 = rng.standard_normal((V, r))
    T = np.array([0.5, 1.0, 2.0])
    x = rng.integers(0, V, (B, g))
    got = draft_lse(L, rng.integers(0, V, B), w1, w2, T, x)
    np.testing.assert_allclose(got, logsumexp(L / T[:, None, None], axis=-1), rtol=1e-13)
    p = draft_distributions(L, np.zeros(B, int), w1, w2, T, x)
    np.testing.assert_allclose(p, np.exp(L / T[:, None, None] - got[..., None]), rtol=1e-12)


def test_residual_gumbel_words_are_the_counters_words():
    seed, off, b, k, V = 0x1234_5678_9ABC, 17, 3, 5, 11
    g = residual_gumbel(seed, off, b, k, V)
    for v in (0, 3, 4, 10):
        w = philox4x32_10(np.uint64(v // 4), np.uint64(b), np.uint64((4 << 16) | k), np.uint64(off),
                          np.uint64(seed & 0xFFFFFFFF), np.uint64(seed >> 32))[v % 4]
        u = ((int(w) >> 9) + 0.5) * 2.0 ** -23
        assert g[v] == pytest.approx(-np.log(-np.log(u)), rel=1e-15)


def test_target_depends_only_on_logits_over_temperature_and_margins():
    t, L, w1, w2, a = _case(5)
    B = 40
    tb, Lb, anchor = _batch(t, L, a, B)
    x = np.random.default_rng(0).integers(0, 6, (B, 2))
    ra = verify_from_logits(tb, np.full(B, 1.0), Lb, anchor, w1, w2, np.ones(B), x, None, 3, 0)
    rb = verify_from_logits(2 * tb, np.full(B, 2.0), Lb, anchor, w1, w2, np.ones(B), x, None, 3, 0)
    np.testing.assert_array_equal(ra[0], rb[0])
    assert np.all(ra[2] > 0) and np.all(ra[3] > 0)


def test_lengths_truncate_and_bonus_comes_from_row_L():
    t, L, w1, w2, a = _case(6)
    B = 200
    tb, Lb, anchor = _batch(t, L, a, B)
    x, _, _ = markov_sample(Lb, anchor, w1, w2, np.ones(B), 1, 0)
    lengths = np.zeros(B, np.int64)
    out, nacc, am, _ = verify_from_logits(tb, np.ones(B), Lb, anchor, w1, w2, np.ones(B), x, lengths, 2, 0)
    assert np.all(nacc == 0) and np.all(out[:, 1:] == -1) and np.all(np.isinf(am))
    # with L_b = 0 the only token is a draw from target row 0
    assert _chi2_ok(out[:, 0], _target_law(t[0], 1.0), 6) > 1e-4
