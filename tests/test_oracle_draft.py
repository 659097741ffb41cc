"""Pins for the oracle's draft step: base logits and sequential Markov sampling.

Checks against closed forms, special cases that reduce to library routines,
brute force on tiny inputs and the sampling law of the Gumbel-max trick
("DSpark implementation and evaluation" §2.2, §3).
"""
import numpy as np
import pytest
from scipy import special, stats

import oracle
from oracle.draft import markov_sample_given_noise
from workloads import DRAFT_CONFIGS, draft_inputs


def test_draft_logits_one_hot_rows_select_lm_head_columns():
    rng = np.random.default_rng(0)
    W = rng.standard_normal((50, 12))
    X = np.zeros((5, 12))
    cols = [0, 3, 11, 7, 3]
    X[np.arange(5), cols] = 1.0
    L = oracle.draft_logits(X, W)
    np.testing.assert_array_equal(L, W[:, cols].T)


def test_draft_logits_small_integers_exact_brute_force():
    rng = np.random.default_rng(1)
    X = rng.integers(-8, 9, size=(3, 7))
    W = rng.integers(-8, 9, size=(5, 7))
    L = oracle.draft_logits(X, W)
    for m in range(3):
        for v in range(5):
            assert L[m, v] == sum(int(X[m, h]) * int(W[v, h]) for h in range(7))


def test_markov_bias_one_hot_embedding_is_a_column_of_w2():
    rng = np.random.default_rng(2)
    V, r = 40, 6
    w1 = np.zeros((V, r))
    w1[np.arange(V), np.arange(V) % r] = 1.0      # token t embeds to e_{t mod r}
    w2 = rng.standard_normal((V, r))
    prev = np.array([0, 13, 39])
    bias = oracle.markov_bias(prev, w1, w2)
    np.testing.assert_array_equal(bias, w2[:, prev % r].T)


def test_markov_bias_zero_embedding_gives_zero_bias():
    w2 = np.random.default_rng(3).standard_normal((30, 4))
    assert np.all(oracle.markov_bias(np.array([5, 6]), np.zeros((30, 4)), w2) == 0)


def test_greedy_is_argmax_of_base_plus_bias_chain():
    """T = 0: no noise; each step is numpy's argmax of base + w2 w1[prev]."""
    rng = np.random.default_rng(4)
    B, N, V, r = 3, 6, 50, 5
    L = rng.standard_normal((B, N, V))
    w1 = rng.standard_normal((V, r))
    w2 = rng.standard_normal((V, r))
    anchor = np.array([1, 2, 3])
    tok, gap, _ = oracle.markov_sample(L, anchor, w1, w2, np.zeros(B), seed=0, offset=0)
    for b in range(B):
        prev = anchor[b]
        for i in range(N):
            expect = int(np.argmax(L[b, i] + np.einsum("vk,k->v", w2, w1[prev])))
            assert tok[b, i] == expect
            prev = expect
    assert np.all(gap >= 0)


def test_ties_go_to_lowest_index():
    V = 10
    L = np.zeros((1, 2, V))
    L[0, 0, [3, 7]] = 5.0
    L[0, 1, [2, 9]] = 5.0
    tok, gap, _ = oracle.markov_sample(L, np.array([0]), np.zeros((V, 2)), np.zeros((V, 2)),
                                       np.zeros(1), 0, 0)
    assert tok.tolist() == [[3, 2]] and np.all(gap == 0)


def test_zero_markov_bias_reduces_to_independent_gumbel_max_softmax_law():
    """w1 = 0: each position is an independent draw from softmax(base / T)."""
    rng = np.random.default_rng(5)
    trials, N, V, T = 400_000, 3, 8, 0.7
    base = rng.standard_normal((N, V)) * 1.5
    L = np.broadcast_to(base, (trials, N, V))
    tok, _, _ = oracle.markov_sample(L, np.zeros(trials, np.int64), np.zeros((V, 2)),
                                     rng.standard_normal((V, 2)), np.full(trials, T), 7, 0)
    for i in range(N):
        p = special.softmax(base[i] / T)
        counts = np.bincount(tok[:, i], minlength=V)
        assert stats.chisquare(counts, p * trials).pvalue > 0.01
    # independence of positions 0 and 1
    joint = np.bincount(tok[:, 0] * V + tok[:, 1], minlength=V * V)
    expect = np.outer(special.softmax(base[0] / T), special.softmax(base[1] / T)).ravel() * trials
    assert stats.chisquare(joint, expect).pvalue > 0.01


@pytest.mark.slow
def test_joint_of_first_two_tokens_matches_markov_chain_law():
    """10^6 trials at V=8: P(x0, x1) = softmax(z0)[x0] * softmax(z1 | x0)[x1] with
    z0 = (L0 + w2 w1[anchor]) / T and z1|x0 = (L1 + w2 w1[x0]) / T."""
    rng = np.random.default_rng(6)
    trials, V, r, T = 1_000_000, 8, 3, 1.0
    base = rng.standard_normal((2, V))
    w1 = rng.standard_normal((V, r)) * 1.5
    w2 = rng.standard_normal((V, r))
    anchor = 5
    L = np.broadcast_to(base, (trials, 2, V))
    tok, _, _ = oracle.markov_sample(L, np.full(trials, anchor), w1, w2, np.full(trials, T), 11, 3)
    p0 = special.softmax((base[0] + w2 @ w1[anchor]) / T)
    expect = np.empty((V, V))
    for x0 in range(V):
        expect[x0] = p0[x0] * special.softmax((base[1] + w2 @ w1[x0]) / T)
    joint = np.bincount(tok[:, 0] * V + tok[:, 1], minlength=V * V)
    assert stats.chisquare(joint, expect.ravel() * trials).pvalue > 0.01
    # and the Markov dependence is real: the law differs from the product of marginals
    marg1 = expect.sum(axis=0)
    assert np.abs(expect - np.outer(p0, marg1)).max() > 1e-2


def test_lse_is_logsumexp_of_scaled_logits():
    rng = np.random.default_rng(7)
    B, N, V, r = 2, 3, 20, 4
    L = rng.standard_normal((B, N, V))
    w1, w2 = rng.standard_normal((V, r)), rng.standard_normal((V, r))
    T = np.array([0.5, 0.0])
    tok, _, lse = oracle.markov_sample(L, np.array([3, 4]), w1, w2, T, 1, 2)
    for b in range(B):
        prev = [3, 4][b]
        for i in range(N):
            logits = L[b, i] + w2 @ w1[prev]
            scale = T[b] if T[b] > 0 else 1.0
            np.testing.assert_allclose(lse[b, i], special.logsumexp(logits / scale), rtol=1e-13)
            prev = tok[b, i]


def test_hand_worked_example(golden_dir):
    """tests/golden/markov_worked.txt: a 2-step, V=3, r=1 case worked out by hand."""
    ex = _read_golden(golden_dir / "markov_worked.txt")
    L = np.array(ex["base"], dtype=np.float64).reshape(1, 2, 3)
    w1 = np.array(ex["w1"], dtype=np.float64).reshape(3, 1)
    w2 = np.array(ex["w2"], dtype=np.float64).reshape(3, 1)
    g = np.array(ex["gumbel"], dtype=np.float64).reshape(2, 3)
    tok, gap, _ = markov_sample_given_noise(L, np.array([int(ex["anchor"][0])]), w1, w2,
                                            np.array([ex["temperature"][0]]),
                                            lambda i, rows: g[i][None, :])
    assert tok[0].tolist() == [int(t) for t in ex["tokens"]]
    np.testing.assert_allclose(gap[0], ex["gap"], rtol=0, atol=1e-12)


def test_req_ids_select_the_counter_of_each_request():
    """Checking a subset of a batch alone reproduces the batch's own tokens."""
    rng = np.random.default_rng(8)
    B, N, V, r = 6, 4, 64, 4
    L = rng.standard_normal((B, N, V))
    w1, w2 = rng.standard_normal((V, r)), rng.standard_normal((V, r))
    anchor = rng.integers(0, V, B)
    T = np.full(B, 1.0)
    full, _, _ = oracle.markov_sample(L, anchor, w1, w2, T, 9, 1)
    sub = np.array([4, 1])
    part, _, _ = oracle.markov_sample(L[sub], anchor[sub], w1, w2, T[sub], 9, 1, req_ids=sub)
    np.testing.assert_array_equal(part, full[sub])


def test_teacher_forced_greedy_steps_are_argmax_on_the_forced_history():
    """Teacher forcing at T = 0: step i is numpy's argmax of base + w2 w1[p_i] with p_0 the anchor
    and p_i the FORCED token of step i - 1 (not the loop's own), written out directly."""
    rng = np.random.default_rng(12)
    B, N, V, r = 4, 5, 40, 3
    L = rng.standard_normal((B, N, V))
    w1, w2 = rng.standard_normal((V, r)) * 2.0, rng.standard_normal((V, r))
    anchor = rng.integers(0, V, B)
    forced = rng.integers(0, V, (B, N))
    tok, gap, lse = oracle.markov_sample(L, anchor, w1, w2, np.zeros(B), 0, 0, forced_tokens=forced)
    for b in range(B):
        for i in range(N):
            p = anchor[b] if i == 0 else forced[b, i - 1]
            logits = L[b, i] + w2 @ w1[p]
            assert tok[b, i] == int(np.argmax(logits))
            srt = np.sort(logits)
            np.testing.assert_allclose(gap[b, i], srt[-1] - srt[-2], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b, i], special.logsumexp(logits), rtol=1e-13)
    # the forced history is used: forcing other tokens changes some step's result
    free, _, _ = oracle.markov_sample(L, anchor, w1, w2, np.zeros(B), 0, 0)
    assert np.any(free[:, 1:] != tok[:, 1:])


def test_teacher_forced_with_zero_markov_head_ignores_the_history():
    """w1 = 0: no step depends on the previous token, so any forced history gives the
    free-running tokens (independent Gumbel-max per position)."""
    rng = np.random.default_rng(13)
    B, N, V, r = 3, 6, 100, 4
    L = rng.standard_normal((B, N, V))
    w1, w2 = np.zeros((V, r)), rng.standard_normal((V, r))
    anchor = rng.integers(0, V, B)
    T = np.array([0.7, 1.0, 1.4])
    free, _, _ = oracle.markov_sample(L, anchor, w1, w2, T, 5, 2)
    forced, _, _ = oracle.markov_sample(L, anchor, w1, w2, T, 5, 2, forced_tokens=rng.integers(0, V, (B, N)))
    np.testing.assert_array_equal(forced, free)


def test_tiny_workload_runs_and_param_count_of_markov_head():
    cfg = DRAFT_CONFIGS["tiny"]
    inp = draft_inputs(cfg)
    L = oracle.draft_logits(inp["hidden_f32"], inp["lm_head_f32"]).reshape(cfg.B, cfg.N, cfg.V)
    tok, gap, _ = oracle.markov_sample(L, inp["anchor"], inp["w1_f32"], inp["w2_f32"],
                                       np.ones(cfg.B), 0, 0)
    assert tok.shape == (1, 8) and np.all((tok >= 0) & (tok < cfg.V))
    # "DSpark implementation and evaluation" §3: 2 * V * r parameters, ~19.4M at V=151936, r=64
    assert 2 * 151936 * 64 == 19_447_808


def _read_golden(path):
    out = {}
    for line in path.read_text().splitlines():
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, vals = line.split(":", 1)
        out[key.strip()] = [float(v) for v in vals.split()]
    return out
