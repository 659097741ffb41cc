"""Pins for the oracle's speculative verification.

Checks against hand-worked cases, the lossless law (the emitted tokens follow
the target distribution exactly), acceptance = 1 - TV, and the degenerate cases
("Speculative decoding: from zero to DSpark" §2).
"""
import numpy as np
import pytest
from scipy import stats

import oracle
from oracle.verify import verify_given_draws, acceptance_probability_exact
from workloads import VERIFY_CONFIGS, verify_inputs


def _read_cases(path):
    rows, cases = {}, []
    for line in path.read_text().splitlines():
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, val = line.split(":", 1)
        key = key.strip()
        if key == "case":
            u, R, L, out, nacc = (p.split() for p in val.split(";"))
            cases.append(dict(u=[float(v) for v in u], R=int(R[0]), L=int(L[0]),
                              out=[int(v) for v in out], nacc=int(nacc[0])))
        elif key == "x":
            rows["x"] = [int(v) for v in val.split()]
        else:
            rows[key] = [[float(v) for v in grp.split()] for grp in val.split("|")]
    return rows, cases


def test_hand_worked_cases(golden_dir):
    rows, cases = _read_cases(golden_dir / "verify_worked.txt")
    p_t = np.array(rows["p_t"], dtype=np.float32)[None]
    p_d = np.array(rows["p_d"], dtype=np.float32)[None]
    x = np.array(rows["x"])[None]
    assert len(cases) == 6
    for c in cases:
        u = np.array([c["u"]], dtype=np.float32)
        R = np.array([[c["R"]] * 3], dtype=object)
        out, nacc, _, numeric = verify_given_draws(p_t, p_d, x, np.array([c["L"]]), u, R)
        assert out[0].tolist() == c["out"], c
        assert nacc[0] == c["nacc"] and not numeric[0]


def _random_pair(rng, V, conc=1.0):
    p_t = rng.dirichlet(np.full(V, conc)).astype(np.float32)
    p_d = rng.dirichlet(np.full(V, conc)).astype(np.float32)
    return p_t, p_d


def _trials(p_t_rows, p_d_rows, trials, seed):
    """Broadcast one block of rows over `trials` requests, draft tokens drawn from p_d."""
    g, V = p_d_rows.shape
    rng = np.random.default_rng(seed)
    x = np.empty((trials, g), dtype=np.int64)
    for k in range(g):
        pk = p_d_rows[k].astype(np.float64)
        x[:, k] = rng.choice(V, size=trials, p=pk / pk.sum())
    P_t = np.broadcast_to(p_t_rows, (trials, g + 1, V))
    P_d = np.broadcast_to(p_d_rows, (trials, g, V))
    return P_t, P_d, x


@pytest.mark.slow
def test_lossless_first_two_emitted_tokens_follow_target():
    """10^6 trials at V=8: the first emitted token ~ p_t[0]; given x_0 accepted the
    second ~ p_t[1]; jointly (o_0, o_1) ~ p_t[0] x p_t[1] when both are emitted."""
    rng = np.random.default_rng(10)
    V, g, trials = 8, 3, 1_000_000
    rows = [_random_pair(rng, V) for _ in range(g + 1)]
    p_t = np.stack([r[0] for r in rows])
    p_d = np.stack([r[1] for r in rows[:g]])
    P_t, P_d, x = _trials(p_t, p_d, trials, 11)
    out, nacc, _, numeric = oracle.verify(P_t, P_d, x, None, seed=2, offset=0)
    assert not numeric.any()
    pt64 = p_t.astype(np.float64) / p_t.astype(np.float64).sum(axis=1, keepdims=True)
    c0 = np.bincount(out[:, 0], minlength=V)
    assert stats.chisquare(c0, pt64[0] * trials).pvalue > 0.01
    both = nacc >= 1
    c01 = np.bincount(out[both, 0] * V + out[both, 1], minlength=V * V)
    # x_0 accepted has law min(p_t, p_d) / (1 - TV); given that, o_1 ~ p_t[1]
    acc0 = np.minimum(p_d[0].astype(np.float64), pt64[0])
    expect = np.outer(acc0 / acc0.sum(), pt64[1]).ravel() * both.sum()
    assert stats.chisquare(c01, expect).pvalue > 0.01


def test_acceptance_probability_is_one_minus_total_variation_exactly():
    """Exact count over the discretised uniforms: sum_x p_d(x) P(accept x) = sum min(p_t, p_d)."""
    rng = np.random.default_rng(12)
    V = 8
    for conc in (0.3, 1.0, 5.0):
        p_t, p_d = _random_pair(rng, V, conc)
        acc = sum(float(p_d[x]) * acceptance_probability_exact(p_t[x], p_d[x]) for x in range(V))
        one_minus_tv = float(np.minimum(p_t.astype(np.float64), p_d.astype(np.float64)).sum())
        assert abs(acc - one_minus_tv) <= V * 2.0 ** -22, (acc, one_minus_tv)


def test_empirical_acceptance_rate_within_four_sigma():
    rng = np.random.default_rng(13)
    V, trials = 8, 200_000
    p_t, p_d = _random_pair(rng, V)
    P_t, P_d, x = _trials(np.stack([p_t, p_t]), p_d[None], trials, 14)
    _, nacc, _, _ = oracle.verify(P_t, P_d, x, None, seed=5, offset=1)
    a = float(np.minimum(p_t, p_d).astype(np.float64).sum())
    rate = nacc.mean()
    assert abs(rate - a) <= 4 * np.sqrt(a * (1 - a) / trials), (rate, a)


def test_identical_distributions_always_accept():
    rng = np.random.default_rng(15)
    V, g, trials = 16, 5, 20_000
    p = np.stack([_random_pair(rng, V)[0] for _ in range(g + 1)])
    P_t, P_d, x = _trials(p, p[:g], trials, 16)
    out, nacc, acc, _ = oracle.verify(P_t, P_d, x, None, seed=1, offset=0)
    assert np.all(nacc == g) and np.all(acc == 1)
    np.testing.assert_array_equal(out[:, :g], x)
    assert np.all(p[g][out[:, g]] > 0)


def test_disjoint_supports_always_reject_into_target_support():
    V, trials = 8, 5_000
    p_t = np.zeros((3, V), np.float32)
    p_t[:, :4] = 0.25
    p_d = np.zeros((2, V), np.float32)
    p_d[:, 4:] = 0.25
    P_t, P_d, x = _trials(p_t, p_d, trials, 17)
    out, nacc, acc, _ = oracle.verify(P_t, P_d, x, None, seed=3, offset=0)
    assert np.all(nacc == 0) and np.all(acc[:, 0] == 0) and np.all(acc[:, 1] == -1)
    assert np.all(out[:, 0] < 4) and np.all(out[:, 1:] == -1)


def test_zero_draft_probability_token_is_accepted_iff_target_positive():
    p_t = np.array([[0.5, 0.5, 0.0], [0.2, 0.3, 0.5]], np.float32)[None]
    p_d = np.array([[0.0, 1.0, 0.0]], np.float32)[None]
    for tok, expect in ((0, 1), (2, 0)):
        _, nacc, _, _ = oracle.verify(p_t, p_d, np.array([[tok]]), None, 0, 0)
        assert nacc[0] == expect


def test_lengths_truncate_the_block():
    rng = np.random.default_rng(18)
    V, g, B = 32, 6, 200
    p = np.stack([_random_pair(rng, V)[0] for _ in range(g + 1)])
    P_t, P_d, x = _trials(p, p[:g], B, 19)
    L = rng.integers(0, g + 1, B)
    out, nacc, acc, _ = oracle.verify(P_t, P_d, x, L, seed=4, offset=0)
    np.testing.assert_array_equal(nacc, L)                     # p_t == p_d accepts all tested
    assert np.all((acc == -1) == (np.arange(g)[None] >= L[:, None]))
    for b in range(B):
        assert out[b, L[b]] >= 0 and np.all(out[b, L[b] + 1:] == -1)


def test_residual_with_no_mass_falls_back_to_target_row():
    # rejected token 3 with p_t <= p_d everywhere: the residual is all zero, so the
    # correction is drawn from the p_t row itself; R = 2^63 picks the middle of its mass
    p_d = np.array([[0.25, 0.25, 0.25, 0.25 + 2 ** -20]], np.float32)[None]
    p_t = np.array([[0.25, 0.25, 0.25, 0.25 - 2 ** -20], [1, 0, 0, 0]], np.float32)[None]
    u = np.array([[1.0 - 2.0 ** -24]], np.float32)
    out, nacc, _, numeric = verify_given_draws(p_t, p_d, np.array([[3]]), None, u,
                                               np.array([[2 ** 63, 0]], dtype=object))
    # Q = 2^40 - 2^20, t = 2^39 - 2^19, prefix (2^38, 2^39, ...) -> token 1
    assert nacc[0] == 0 and not numeric[0] and out[0].tolist() == [1, -1]


def test_target_row_without_mass_gives_argmax_and_numeric_flag():
    p_d = np.array([[0.5, 0.5, 0.0]], np.float32)[None]
    p_t = np.array([[0.0, 0.0, 0.0], [0.2, 0.3, 0.5]], np.float32)[None]
    out, nacc, acc, numeric = oracle.verify(p_t, p_d, np.array([[1]]), None, 0, 0)
    assert nacc[0] == 0 and acc[0, 0] == 0 and numeric[0] and out[0].tolist() == [0, -1]


def test_workload_generator_shapes_tiny():
    inp = verify_inputs(VERIFY_CONFIGS["tiny"])
    assert inp["p_t"].shape == (1, 9, 4096) and inp["p_d"].shape == (1, 8, 4096)
    np.testing.assert_allclose(inp["p_t"].sum(-1), 1, rtol=1e-5)
    out, nacc, _, numeric = oracle.verify(inp["p_t"], inp["p_d"], inp["draft_tokens"], None, 2, 0)
    assert 0 <= nacc[0] <= 8 and not numeric.any()
