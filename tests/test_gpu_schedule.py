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
