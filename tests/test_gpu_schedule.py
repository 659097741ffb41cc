"""GPU parity: confidence-scheduled admission against the oracle, bit for bit.

Survival (fp32 chain), the chosen K (fixed-point sums, one fp64 multiply per K),
the admitted set in rank order and the per-request lengths must all be equal.
"""
import numpy as np
import pytest

import oracle
from tests._helpers import to_dev
from workloads import SCHEDULE_CONFIGS, schedule_inputs, sps_table

pytestmark = pytest.mark.gpu


def _check(ds, c, sps, K_in):
    ws = ds.Workspace(ds.OP_SCHEDULE, c.shape[0], c.shape[1])
    surv, K, lengths, sel = ds.dspark_schedule(to_dev(c), None if sps is None else to_dev(sps), K_in,
                                               workspace=ws)
    st, bits = ds.dspark_read_status(ws)
    ref = oracle.schedule(c, sps, K_in)
    np.testing.assert_array_equal(surv.cpu().numpy(), ref["survival"])
    assert int(K.item()) == ref["K"]
    np.testing.assert_array_equal(lengths.cpu().numpy(), ref["lengths"])
    np.testing.assert_array_equal(sel.cpu().numpy(), ref["selected"])
    return ref, st, bits


def test_tiny_fixed_K(cuda_lib):
    cfg = SCHEDULE_CONFIGS["tiny"]
    inp = schedule_inputs(cfg)
    ref, st, _ = _check(cuda_lib, inp["cond_accept"], inp["sps"], cfg.K_in)
    assert ref["K"] == 6 and st == 0


def test_schedule_workload_full_size(cuda_lib):
    """B=1024, N=16, SPS over 1..16384 with a sawtooth: K chosen by full scan."""
    cfg = SCHEDULE_CONFIGS["schedule"]
    inp = schedule_inputs(cfg)
    ref, st, _ = _check(cuda_lib, inp["cond_accept"], inp["sps"], -1)
    assert st == 0
    print(f"schedule: K={ref['K']}, mean length {ref['lengths'].mean():.2f}")


@pytest.mark.parametrize("trial", range(12))
def test_random_small_cases(cuda_lib, trial):
    rng = np.random.default_rng(100 + trial)
    B = int(rng.integers(1, 300))
    N = int(rng.integers(1, 20))
    c = rng.beta(rng.uniform(0.5, 9), rng.uniform(0.5, 3), size=(B, N)).astype(np.float32)
    if trial % 3 == 0:
        c[rng.random((B, N)) < 0.2] = 1.0          # survival ties
        c[rng.random((B, N)) < 0.05] = 0.0
    S = int(rng.integers(1, B * N + 50))
    sps = sps_table(S) * rng.uniform(0.5, 1.5)
    K_in = -1 if trial % 2 == 0 else int(rng.integers(0, B * N + 10))
    _check(cuda_lib, c, sps if K_in < 0 else None, K_in)


def test_out_of_range_confidences_are_clamped_and_flagged(cuda_lib):
    c = np.array([[0.9, 1.5, 0.5], [np.nan, 0.3, -0.2]], np.float32)
    ref, st, bits = _check(cuda_lib, c, sps_table(6), -1)
    assert ref["clamped"] and bits & cuda_lib.STATUS_INPUT_RANGE


@pytest.mark.parametrize("B,N", [(16, 16), (257, 1), (32, 32), (41, 25), (100, 20), (64, 32), (2049, 1),
                                 (1023, 16), (1, 16384)])
def test_pool_sizes_around_block_and_round_edges(cuda_lib, B, N):
    """Pools at and just past 256, 1024 and 2048 candidates (the bitonic and the radix sort),
    ragged warp runs, the 16384 maximum of the shared-memory sort with a single request."""
    rng = np.random.default_rng(B * 1000 + N)
    c = rng.beta(4, 1.5, size=(B, N)).astype(np.float32)
    c[rng.random((B, N)) < 0.15] = 1.0
    _check(cuda_lib, c, sps_table(B * N), -1)


def test_large_pool_beyond_shared_memory(cuda_lib):
    """B*N = 17600 > 16384: the keys live in the workspace."""
    rng = np.random.default_rng(7)
    c = rng.beta(5, 2, size=(1100, 16)).astype(np.float32)
    c[rng.random(c.shape) < 0.1] = 1.0
    _check(cuda_lib, c, sps_table(16384), -1)
    _check(cuda_lib, c, None, 12345)


@pytest.mark.parametrize("B,N", [(64, 16), (1100, 16)])
def test_objective_with_special_sps_values(cuda_lib, B, N):
    """SPS entries that are zero, subnormal, negative, infinite, NaN, or so large or small that
    the product overflows or leaves the normal range: K must still match the oracle's fp64."""
    rng = np.random.default_rng(11 + B)
    c = rng.beta(3, 1, size=(B, N)).astype(np.float32)
    S = B * N
    sps = sps_table(S).copy()
    specials = np.array([0.0, -0.0, 5e-324, 1e-310, -3.0, np.inf, -np.inf, np.nan, 1e300, 1.7e308,
                         1e-300, 2.2250738585072014e-308 * 1.5], np.float64)
    pos = rng.choice(S, size=S // 4, replace=False)
    sps[pos] = rng.choice(specials, size=pos.size)
    _check(cuda_lib, c, sps, -1)
    # every entry NaN or -inf: nothing beats -inf, K = 1 and the numeric flag is raised
    sps_bad = np.where(rng.random(S) < 0.5, np.nan, -np.inf)
    ref, st, bits = _check(cuda_lib, c, sps_bad, -1)
    assert ref["K"] == 1 and bits & cuda_lib.STATUS_NUMERIC


def test_negative_zero_confidence_is_zero(cuda_lib):
    """-0.0 and +0.0 survivals are one value: ties are broken by position, as for any tie."""
    c = np.array([[0.5, -0.0, 0.7], [0.0, 0.9, 0.3], [-0.0, 0.0, 1.0]], np.float32)
    _check(cuda_lib, c, sps_table(9), -1)
    _check(cuda_lib, c, None, 7)


@pytest.mark.parametrize("B,N", [(1, 1), (1, 8), (4, 8), (32, 1), (3, 10), (2, 16), (1, 32), (5, 6)])
@pytest.mark.parametrize("K_in", [-1, 0, 5, 40])
def test_pools_of_at_most_32_candidates(cuda_lib, B, N, K_in):
    """One-warp pools (a few decode requests), with ties, special SPS entries and fixed K."""
    rng = np.random.default_rng(B * 100 + N + K_in)
    c = rng.beta(3, 1, size=(B, N)).astype(np.float32)
    c[rng.random((B, N)) < 0.3] = 1.0
    c[rng.random((B, N)) < 0.1] = 0.0
    sps = None
    if K_in < 0:
        sps = sps_table(B * N + 3)
        sps[rng.random(sps.size) < 0.2] = np.nan
        sps[rng.random(sps.size) < 0.1] = 0.0
    _check(cuda_lib, c, sps, K_in)


@pytest.mark.parametrize("B,N,case", [(1024, 16, "ties"), (1023, 16, "fixed"), (3, 700, "short_S"), (130, 16, "nan_sps"),
                                      (2049, 1, "clamp"), (300, 10, "fixed0"), (8, 2048, "ties"), (1000, 13, "short_S"),
                                      (517, 31, "negzero")])
def test_pools_sorted_across_a_cluster(cuda_lib, B, N, case):
    """Pools of 2049 .. 16384 candidates whose requests split into eight blocks of at most 2048
    keys are sorted across a thread-block cluster: ragged and empty blocks (B not a multiple of
    eight, B < 8), heavy survival ties across block boundaries, K fixed (0, inside, past the
    pool), S ending inside a block, special SPS entries, clamped and negative-zero inputs."""
    rng = np.random.default_rng(B * 31 + N)
    c = rng.beta(4, 1.5, size=(B, N)).astype(np.float32)
    n = B * N
    sps, K_in = sps_table(n), -1
    if case == "ties":
        c[rng.random((B, N)) < 0.4] = 1.0
        c[rng.random((B, N)) < 0.1] = 0.0
    elif case == "fixed":
        for K_in in (0, 1, n // 3, n, n + 5):
            _check(cuda_lib, c, None, K_in)
        return
    elif case == "fixed0":
        sps, K_in = None, 0
    elif case == "short_S":
        sps = sps_table(n // 2 + 7)
    elif case == "nan_sps":
        sps[rng.random(n) < 0.3] = np.nan
        sps[rng.random(n) < 0.1] = -np.inf
    elif case == "clamp":
        c[rng.random((B, N)) < 0.01] = 1.5
        c[rng.random((B, N)) < 0.01] = np.nan
    elif case == "negzero":
        c[rng.random((B, N)) < 0.2] = -0.0
        c[rng.random((B, N)) < 0.2] = 0.0
    ref, st, bits = _check(cuda_lib, c, sps, K_in)
    if case == "clamp":
        assert bits & cuda_lib.STATUS_INPUT_RANGE
    else:
        assert st == 0
