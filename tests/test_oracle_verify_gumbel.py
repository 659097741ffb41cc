"""Pins of the oracle of verification with the draft's Gumbel noise: a hand-worked case, the
coupling with the sampler (the target scoring the draft's own logits accepts every token), the
law of the emitted tokens (the target's own law at each position, also given the acceptance
of the one before), the temperature-0 case against greedy verification, truncation and
invalid inputs."""
import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import verify_gumbel, target_gumbel_tokens, verify_greedy


def _read(path):
    d = {"cases": []}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, val = line.partition(":")
        val = val.strip()
        if key == "case":
            draft, res = val.split("->")
            out, nacc = res.split(";")
            d["cases"].append((np.array([int(v) for v in draft.split()]),
                               np.array([int(v) for v in out.split()]), int(nacc)))
        else:
            d[key] = np.array([float(v) for v in val.split()])
    return d


def test_hand_worked_case(golden_dir):
    d = _read(golden_dir / "verify_gumbel_worked.txt")
    t = d["target"].reshape(1, 3, 3)
    noise_rows = d["noise"].reshape(3, 3)
    noise = lambda k, req: np.repeat(noise_rows[k][None], len(req), axis=0)
    assert len(d["cases"]) == 2
    for draft, out, nacc in d["cases"]:
        got, n = verify_gumbel(t, d["temperature"], draft[None], 0, 0, noise=noise)
        np.testing.assert_array_equal(got[0], out)
        assert n[0] == nacc


def test_target_scoring_the_drafts_own_logits_accepts_everything():
    # the draft samples with oracle.markov_sample (seed, offset); a target whose row k is exactly
    # the draft's scaled logits at step k (base + Markov bias of its own previous token) and whose
    # temperature is the draft's draws every drafted token again: all accepted, and the bonus is
    # the Gumbel-max of row gamma with the noise of step gamma
    rng = np.random.default_rng(7)
    B, N, V, r = 6, 5, 40, 4
    L = rng.standard_normal((B, N, V)) * 2
    w1 = rng.standard_normal((V, r))
    w2 = rng.standard_normal((V, r)) / 2
    anchor = rng.integers(0, V, B)
    T = np.array([1.0, 0.7, 1.3, 1.0, 0.5, 2.0])
    seed, offset = 11, 3
    x, _, _ = oracle.markov_sample(L, anchor, w1, w2, T, seed, offset)
    prev = np.concatenate([anchor[:, None], x[:, :-1]], axis=1)
    t = np.empty((B, N + 1, V))
    for k in range(N):
        t[:, k] = L[:, k] + oracle.markov_bias(prev[:, k], w1, w2)
    t[:, N] = rng.standard_normal((B, V))
    out, nacc = verify_gumbel(t, T, x, seed, offset)
    assert np.all(nacc == N)
    np.testing.assert_array_equal(out[:, :N], x)
    y, _ = target_gumbel_tokens(t, T, seed, offset)
    np.testing.assert_array_equal(out[:, N], y[:, N])
    # the noise of another offset breaks the coupling: most requests now stop early
    _, nacc2 = verify_gumbel(t, T, x, seed, offset + 1)
    assert nacc2.mean() < N


@pytest.mark.slow
def test_emitted_tokens_follow_the_target_law():
    # 200000 requests, V = 8: draft and target logits differ; the draft's tokens are its own
    # Gumbel-max draws with the shared noise.  The first emitted token follows softmax(t0 / T);
    # given that x0 was accepted, the second follows softmax(t1 / T) (its noise is independent
    # of what decided the first), though x1 was drawn from the draft's logits
    rng = np.random.default_rng(3)
    B, V, T = 200_000, 8, 0.8
    t_row = rng.standard_normal((2, V)) * 1.5
    d_row = t_row + rng.standard_normal((2, V))
    t = np.broadcast_to(np.concatenate([t_row, rng.standard_normal((1, V))])[None], (B, 3, V)).copy()
    Ts = np.full(B, T)
    seed, offset = 5, 9
    x = np.stack([np.argmax(d_row[k] / T + oracle.philox.draft_gumbel(seed, offset, np.arange(B), k, V), axis=1)
                  for k in range(2)], axis=1)
    out, nacc = verify_gumbel(t, Ts, x, seed, offset)

    def law(row):
        p = np.exp(row / T - (row / T).max())
        return p / p.sum()

    counts = np.bincount(out[:, 0], minlength=V)
    assert stats.chisquare(counts, law(t_row[0]) * B).pvalue > 0.01
    acc = nacc >= 1
    counts = np.bincount(out[acc, 1], minlength=V)
    assert stats.chisquare(counts, law(t_row[1]) * acc.sum()).pvalue > 0.01
    # the coupling accepts far more often than independent draws would (sum_v p_t p_d)
    p_ind = float((law(t_row[0]) * law(d_row[0])).sum())
    assert acc.mean() > p_ind + 0.05


def test_temperature_zero_is_greedy_verification():
    rng = np.random.default_rng(1)
    B, g, V = 20, 4, 30
    t = rng.standard_normal((B, g + 1, V))
    x = rng.integers(0, V, (B, g))
    x[:10] = np.argmax(t[:10, :g], axis=2)              # some requests match the argmax chain
    lengths = rng.integers(0, g + 1, B)
    out, nacc = verify_gumbel(t, np.zeros(B), x, 4, 2, lengths)
    out_g, nacc_g = verify_greedy(t, x, lengths)
    np.testing.assert_array_equal(out, out_g)
    np.testing.assert_array_equal(nacc, nacc_g)


def test_truncation_uses_the_row_and_noise_of_the_length():
    rng = np.random.default_rng(2)
    B, g, V = 8, 5, 25
    t = rng.standard_normal((B, g + 1, V))
    T = np.full(B, 1.0)
    y, _ = target_gumbel_tokens(t, T, 6, 0)
    x = y[:, :g].copy()                                  # every drafted token matches
    lengths = np.array([0, 1, 2, 3, 4, 5, 2, 0])
    out, nacc = verify_gumbel(t, T, x, 6, 0, lengths)
    np.testing.assert_array_equal(nacc, lengths)
    for b in range(B):
        L = lengths[b]
        np.testing.assert_array_equal(out[b, :L], x[b, :L])
        assert out[b, L] == y[b, L]
        assert np.all(out[b, L + 1:] == -1)


def test_invalid_requests_and_request_ids():
    rng = np.random.default_rng(4)
    B, g, V = 4, 3, 12
    t = rng.standard_normal((B, g + 1, V))
    x = rng.integers(0, V, (B, g))
    x[1, 0] = V                                          # out-of-range token
    lengths = np.array([3, 3, -1, 4])                    # bad lengths for requests 2 and 3
    out, nacc = verify_gumbel(t, np.ones(B), x, 1, 1, lengths)
    for b in (1, 2, 3):
        assert nacc[b] == 0 and np.all(out[b] == -1)
    assert out[0, nacc[0]] >= 0
    # a subset verified on its own with its draft-batch request ids gives the same rows
    full_out, full_n = verify_gumbel(t[[0, 0, 0]], np.ones(3), x[[0, 0, 0]], 1, 1, req_ids=[0, 1, 2])
    sub_out, sub_n = verify_gumbel(t[[0]], np.ones(1), x[[0]], 1, 1, req_ids=[2])
    np.testing.assert_array_equal(sub_out[0], full_out[2])
