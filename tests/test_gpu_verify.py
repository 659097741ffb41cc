"""GPU parity: lossless speculative verification against the oracle, bit for bit.

Accept/reject decisions and emitted tokens are exact (fp32 ratio test in the
same rounding, integer inverse CDF on both sides).
"""
import numpy as np
import pytest
from scipy import stats

import oracle
from tests._helpers import to_dev
from workloads import VERIFY_CONFIGS, VerifyConfig, verify_inputs

pytestmark = pytest.mark.gpu


def _gpu(ds, p_t, p_d, x, lengths, seed, offset):
    ws = ds.Workspace(ds.OP_VERIFY, p_t.shape[0], p_t.shape[1] - 1, p_t.shape[2])
    out, nacc = ds.dspark_verify(to_dev(p_t), to_dev(p_d), to_dev(np.asarray(x, np.int32)),
                                 None if lengths is None else to_dev(np.asarray(lengths, np.int32)),
                                 seed, offset, workspace=ws)
    st, bits = ds.dspark_read_status(ws)
    return out.cpu().numpy(), nacc.cpu().numpy(), st, bits


def _check_exact(ds, p_t, p_d, x, lengths, seed, offset):
    out, nacc, st, bits = _gpu(ds, p_t, p_d, x, lengths, seed, offset)
    ro, rn, _, rnum = oracle.verify(p_t, p_d, x, lengths, seed, offset)
    np.testing.assert_array_equal(nacc, rn)
    np.testing.assert_array_equal(out, ro)
    return out, nacc, st, bits, rnum


def test_tiny_exact(cuda_lib):
    inp = verify_inputs(VERIFY_CONFIGS["tiny"])
    _, _, st, _, _ = _check_exact(cuda_lib, inp["p_t"], inp["p_d"], inp["draft_tokens"], None, 2, 0)
    assert st == 0


def test_verify_workload_full_size_exact(cuda_lib):
    """B=256, gamma=8, V=151936: every request's decisions and tokens bit-exact."""
    cfg = VERIFY_CONFIGS["verify"]
    inp = verify_inputs(cfg)
    out, nacc, st, _, _ = _check_exact(cuda_lib, inp["p_t"], inp["p_d"], inp["draft_tokens"], None,
                                       cfg.verify_seed, 0)
    assert st == 0
    for s in cfg.draft_sigmas:
        sel = inp["sigma"] == np.float32(s)
        print(f"sigma={s}: mean accepted {nacc[sel].mean():.2f} of {cfg.gamma}")


@pytest.mark.parametrize("V", [1, 5, 1001, 4096, 70001])
def test_ragged_vocab_and_lengths_exact(cuda_lib, V):
    cfg = VerifyConfig("r", B=40, gamma=3, V=V, target_std=1.5, draft_sigmas=(0.5, 2.0),
                       independent_draft=False, data_seed=V)
    inp = verify_inputs(cfg)
    L = np.random.default_rng(V).integers(0, cfg.gamma + 1, cfg.B)
    L[:4] = [0, cfg.gamma, 1, 0]
    _, _, st, _, _ = _check_exact(cuda_lib, inp["p_t"], inp["p_d"], inp["draft_tokens"], L, 9, 3)
    assert st == 0


def _trials(p_t_rows, p_d_rows, trials, seed):
    g, V = p_d_rows.shape
    rng = np.random.default_rng(seed)
    x = np.empty((trials, g), dtype=np.int32)
    for k in range(g):
        pk = p_d_rows[k].astype(np.float64)
        x[:, k] = rng.choice(V, size=trials, p=pk / pk.sum())
    P_t = np.ascontiguousarray(np.broadcast_to(p_t_rows, (trials, g + 1, V)))
    P_d = np.ascontiguousarray(np.broadcast_to(p_d_rows, (trials, g, V)))
    return P_t, P_d, x


def test_lossless_and_acceptance_million_trials(cuda_lib):
    """10^6 requests at V=8: first emitted token ~ p_t[0] (chi-square), acceptance within
    4 sigma of 1 - TV, and every output equal to the oracle's."""
    rng = np.random.default_rng(30)
    V, g, trials = 8, 2, 1_000_000
    p_t = rng.dirichlet(np.ones(V), size=g + 1).astype(np.float32)
    p_d = rng.dirichlet(np.ones(V), size=g).astype(np.float32)
    P_t, P_d, x = _trials(p_t, p_d, trials, 31)
    out, nacc, st, _, _ = _check_exact(cuda_lib, P_t, P_d, x, None, 5, 0)
    assert st == 0
    pt0 = p_t[0].astype(np.float64) / p_t[0].astype(np.float64).sum()
    c0 = np.bincount(out[:, 0], minlength=V)
    assert stats.chisquare(c0, pt0 * trials).pvalue > 0.01
    a = float(np.minimum(p_t[0], p_d[0]).astype(np.float64).sum())
    rate = (nacc >= 1).mean()
    assert abs(rate - a) <= 4 * np.sqrt(a * (1 - a) / trials)


def test_identical_and_disjoint_distributions(cuda_lib):
    V, g, B = 64, 4, 500
    rng = np.random.default_rng(32)
    p = rng.dirichlet(np.ones(V), size=g + 1).astype(np.float32)
    P_t, P_d, x = _trials(p, p[:g], B, 33)
    out, nacc, _, _, _ = _check_exact(cuda_lib, P_t, P_d, x, None, 1, 0)
    assert np.all(nacc == g)
    q_t = np.zeros((g + 1, V), np.float32)
    q_t[:, : V // 2] = 2.0 / V
    q_d = np.zeros((g, V), np.float32)
    q_d[:, V // 2:] = 2.0 / V
    P_t, P_d, x = _trials(q_t, q_d, B, 34)
    out, nacc, _, _, _ = _check_exact(cuda_lib, P_t, P_d, x, None, 1, 0)
    assert np.all(nacc == 0) and np.all(out[:, 0] < V // 2)


def test_zero_mass_and_bad_inputs_set_status(cuda_lib):
    p_d = np.array([[[0.5, 0.5, 0.0, 0.0]]], np.float32)
    p_t = np.array([[[0.0, 0.0, 0.0, 0.0], [0.25, 0.25, 0.25, 0.25]]], np.float32)
    out, nacc, st, bits, rnum = _check_exact(cuda_lib, p_t, p_d, np.array([[1]]), None, 0, 0)
    assert rnum[0] and bits & cuda_lib.STATUS_NUMERIC and out[0].tolist() == [0, -1]
    out, nacc, st, bits = _gpu(cuda_lib, p_t, p_d, np.array([[7]]), None, 0, 0)
    assert bits & cuda_lib.STATUS_INPUT_RANGE and nacc[0] == 0 and np.all(out == -1)
    out, nacc, st, bits = _gpu(cuda_lib, p_t, p_d, np.array([[1]]), np.array([2]), 0, 0)
    assert bits & cuda_lib.STATUS_INPUT_RANGE


@pytest.mark.parametrize("V", [700, 151936])
def test_sparse_rows_with_signed_zeros_exact(cuda_lib, V):
    """Rows where most entries are +0 or -0 (top-k truncated distributions): a -0 probability has
    no mass, exactly as +0; the residual often lives in a handful of segments."""
    rng = np.random.default_rng(V + 17)
    B, g = 24, 5
    p_t = np.zeros((B, g + 1, V), np.float32)
    p_d = np.zeros((B, g, V), np.float32)
    for b in range(B):
        for k in range(g + 1):
            sup = rng.choice(V, size=8, replace=False)
            w = rng.random(8).astype(np.float32)
            p_t[b, k, sup] = w / w.sum()
            if k < g:
                sup_d = np.concatenate([sup[:4], rng.choice(V, size=4, replace=False)])
                wd = rng.random(8).astype(np.float32)
                p_d[b, k, sup_d] = wd / wd.sum()
    neg = rng.random(p_t.shape) < 0.3
    p_t[neg & (p_t == 0)] = -0.0
    negd = rng.random(p_d.shape) < 0.3
    p_d[negd & (p_d == 0)] = -0.0
    x = np.empty((B, g), np.int32)
    for b in range(B):
        for k in range(g):
            pk = np.abs(p_d[b, k]).astype(np.float64)
            x[b, k] = rng.choice(V, p=pk / pk.sum())
    _check_exact(cuda_lib, p_t, p_d, x, None, 31, 4)
