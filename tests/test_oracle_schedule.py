"""Pins for the oracle's confidence-scheduled admission.

Checks against brute-force enumeration of every prefix-closed allocation on
tiny inputs, monotone survival, non-anticipation and the full-K search
("Speculative decoding: from zero to DSpark" §6, §7).
"""
import itertools

import numpy as np

import oracle
from oracle.schedule import survival_chain
from workloads import SCHEDULE_CONFIGS, schedule_inputs, sps_table


def _brute_force(c, sps):
    """Best allocation over all (L_0..L_{B-1}) in [0, N]^B with 1 <= sum L <= min(B*N, S).

    Value of an allocation = (B * 2^32 + sum of floor(s * 2^32) over admitted
    prefixes) * SPS[K - 1], K = sum L; returns (best K, best fixed-point sum per K).
    """
    s, _ = survival_chain(c)
    B, N = s.shape
    q = np.floor(s.astype(np.float64) * 2.0 ** 32).astype(np.int64)
    best_sum = {}
    for L in itertools.product(range(N + 1), repeat=B):
        K = sum(L)
        if K == 0 or K > min(B * N, len(sps)):
            continue
        tot = sum(int(q[b, :L[b]].sum()) for b in range(B))
        best_sum[K] = max(best_sum.get(K, -1), tot)
    best_f, best_K = -np.inf, None
    for K in sorted(best_sum):
        f = float(B * 2 ** 32 + best_sum[K]) * float(sps[K - 1])
        if f > best_f:
            best_f, best_K = f, K
    return best_K, best_sum


def test_brute_force_over_prefix_closed_allocations():
    rng = np.random.default_rng(20)
    for trial in range(150):
        B = int(rng.integers(1, 4))
        N = int(rng.integers(1, 4))
        c = rng.random((B, N)).astype(np.float32)
        if trial % 5 == 0:
            c[rng.random((B, N)) < 0.3] = np.float32(1.0)      # ties in survival
        S = int(rng.integers(1, B * N + 2))
        sps = rng.random(S) * 10 + 1
        res = oracle.schedule(c, sps, -1)
        K_bf, best_sum = _brute_force(c, sps)
        assert res["K"] == K_bf, (trial, res["K"], K_bf)
        s = res["survival"]
        q = np.floor(s.astype(np.float64) * 2.0 ** 32).astype(np.int64)
        got = sum(int(q[b, :res["lengths"][b]].sum()) for b in range(B))
        assert got == best_sum[K_bf]
        assert res["lengths"].sum() == K_bf


def test_selection_is_prefix_closed_and_lengths_match():
    rng = np.random.default_rng(21)
    c = rng.beta(2, 1, size=(40, 9)).astype(np.float32)
    c[3, 2] = 1.0
    c[7] = 1.0
    for K_in in (0, 1, 17, 200, 360, 1000):
        res = oracle.schedule(c, None, K_in)
        K = min(K_in, 360)
        assert res["K"] == K
        sel = res["selected"]
        assert np.all(sel[K:] == -1) and len(set(sel[:K].tolist())) == K
        taken = np.zeros((40, 9), bool)
        taken.reshape(-1)[sel[:K]] = True
        for b in range(40):
            Lb = res["lengths"][b]
            assert taken[b, :Lb].all() and not taken[b, Lb:].any()


def test_survival_is_monotone_and_matches_products():
    rng = np.random.default_rng(22)
    c = rng.random((500, 16)).astype(np.float32)
    s, clamped = survival_chain(c)
    assert not clamped
    assert np.all(np.diff(s, axis=1) <= 0)
    np.testing.assert_allclose(s, np.cumprod(c.astype(np.float64), axis=1), rtol=1e-5)
    s2, clamped2 = survival_chain(np.array([[1.5, -0.1, np.nan]], np.float32))
    assert clamped2 and s2.tolist() == [[1.0, 0.0, 0.0]]


def test_non_anticipation_admission_ignores_later_positions():
    """With K fixed, admission of (b, k) does not change when c_{b, j>k} change."""
    rng = np.random.default_rng(23)
    B, N, K = 30, 8, 70
    c = rng.beta(3, 1, size=(B, N)).astype(np.float32)
    base = oracle.schedule(c, None, K)["lengths"]
    for trial in range(200):
        b = int(rng.integers(0, B))
        k = int(rng.integers(0, N))
        c2 = c.copy()
        c2[b, k + 1:] = rng.random(N - k - 1).astype(np.float32)
        L2 = oracle.schedule(c2, None, K)["lengths"]
        assert (base[b] > k) == (L2[b] > k)


def test_full_scan_finds_global_optimum_past_a_local_one():
    # sawtooth SPS: an early-stopping search would halt at the first drop
    c = np.full((4, 8), 0.97, np.float32)
    sps = np.ones(32)
    sps[4] = 0.5          # K = 5 drops ...
    sps[20:] = 1.6        # ... but K = 32 is better
    res = oracle.schedule(c, sps, -1)
    assert res["K"] == 32


def test_schedule_workload_runs():
    cfg = SCHEDULE_CONFIGS["schedule"]
    inp = schedule_inputs(cfg, B=64)
    res = oracle.schedule(inp["cond_accept"], inp["sps"], -1)
    assert 1 <= res["K"] <= 64 * 16
    sps = sps_table(16384)
    assert sps.shape == (16384,) and abs(sps[0] - 105.0) < 1e-9 and abs(sps[127] - 95.0) < 1e-9
