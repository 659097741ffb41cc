"""GPU parity: greedy (temperature-0) verification against the oracle, bit for bit.

Draft tokens are the target's argmax at each position with a per-request probability (so
acceptance lengths vary), otherwise another token; rows are probabilities or logits, with
ties, NaN entries, ragged vocabularies, truncated blocks and invalid requests.
"""
import numpy as np
import pytest

import oracle
from tests._helpers import to_dev
from workloads import VERIFY_CONFIGS, verify_inputs

pytestmark = pytest.mark.gpu


def _drafts(target, p_follow, seed):
    rng = np.random.default_rng(seed)
    B, g1, V = target.shape
    am = np.argmax(np.where(np.isnan(target), -np.inf, target), axis=2)[:, :g1 - 1]
    other = (am + rng.integers(1, max(2, V), size=am.shape)) % V
    follow = rng.random(am.shape) < np.asarray(p_follow)[:, None]
    return np.where(follow, am, other).astype(np.int32)


def _check(ds, target, x, lengths=None):
    out, nacc = ds.dspark_verify_greedy(to_dev(target), to_dev(x), None if lengths is None else to_dev(lengths))
    ref_out, ref_nacc = oracle.verify_greedy(target, x, lengths)
    np.testing.assert_array_equal(nacc.cpu().numpy(), ref_nacc)
    np.testing.assert_array_equal(out.cpu().numpy(), ref_out)
    return ref_nacc


def test_verify_workload_full_size(cuda_lib):
    """B=256, gamma=8, V=151936 target probabilities; acceptance from 0 to 8."""
    inp = verify_inputs(VERIFY_CONFIGS["verify"])
    t = inp["p_t"]
    x = _drafts(t, np.linspace(0.2, 1.0, t.shape[0]), 1)
    nacc = _check(cuda_lib, t, x)
    assert nacc.min() == 0 and nacc.max() == 8


@pytest.mark.parametrize("V", [1, 5, 1001, 2047, 2048, 2049, 70001])
def test_ragged_vocab_ties_and_lengths(cuda_lib, V):
    rng = np.random.default_rng(V)
    B, gamma = 37, 5
    t = rng.integers(0, 3, size=(B, gamma + 1, V)).astype(np.float32)     # many ties
    x = _drafts(t, rng.random(B), V + 1)
    lengths = rng.integers(0, gamma + 1, B).astype(np.int32)
    _check(cuda_lib, t, x, lengths)


def test_logits_and_probabilities_agree(cuda_lib):
    rng = np.random.default_rng(2)
    logits = (rng.standard_normal((16, 9, 30000)) * 3).astype(np.float32)
    x = _drafts(logits, np.full(16, 0.8), 3)
    a, na = cuda_lib.dspark_verify_greedy(to_dev(logits), to_dev(x))
    _check(cuda_lib, logits, x)
    m = logits.max(axis=2, keepdims=True)
    p = np.exp(logits - m)
    p = (p / p.sum(axis=2, keepdims=True)).astype(np.float32)
    # softmax in fp32 can merge near-equal logits into ties; compare where the argmax survives
    same = np.all(np.argmax(p, axis=2) == np.argmax(logits, axis=2), axis=1)
    b, nb = cuda_lib.dspark_verify_greedy(to_dev(p), to_dev(x))
    np.testing.assert_array_equal(a.cpu().numpy()[same], b.cpu().numpy()[same])


def test_nan_rows_and_invalid_requests(cuda_lib):
    rng = np.random.default_rng(5)
    B, gamma, V = 6, 4, 3000
    t = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    t[0, 1, ::3] = np.nan
    t[1, 2, :] = np.nan                                  # no entry at all: token 0, NUMERIC
    x = _drafts(t, np.ones(B), 7)
    x[1, 2] = 0
    x[3, 1] = V + 2                                      # invalid token
    lengths = np.array([4, 4, 4, 4, 9, -1], np.int32)    # two invalid lengths
    import torch
    ws = cuda_lib.Workspace(cuda_lib.OP_VERIFY_GREEDY, B, gamma)
    out, nacc = cuda_lib.dspark_verify_greedy(to_dev(t), to_dev(x), to_dev(lengths), workspace=ws)
    st, bits = cuda_lib.dspark_read_status(ws)
    ref_out, ref_nacc = oracle.verify_greedy(t, x, lengths)
    np.testing.assert_array_equal(out.cpu().numpy(), ref_out)
    np.testing.assert_array_equal(nacc.cpu().numpy(), ref_nacc)
    assert bits & cuda_lib.STATUS_INPUT_RANGE and bits & cuda_lib.STATUS_NUMERIC


def test_many_small_requests_share_warps(cuda_lib):
    rng = np.random.default_rng(9)
    B, gamma, V = 3000, 3, 64
    t = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    x = _drafts(t, rng.random(B), 11)
    _check(cuda_lib, t, x, rng.integers(0, gamma + 1, B).astype(np.int32))
