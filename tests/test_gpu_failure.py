"""Failure detection on the GPU without a fault: a bounded device wait that runs out
records TIMEOUT in the workspace status word and the context stays usable."""
import numpy as np
import pytest

import oracle
from tests._helpers import to_dev
from workloads import SCHEDULE_CONFIGS, schedule_inputs

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_context_survives(cuda_lib):
    import time
    import torch
    ds = cuda_lib
    ws = ds.Workspace(ds.OP_VERIFY)
    t0 = time.time()
    ds.dspark_selftest_wait_timeout(ws, 20_000_000)          # 20 ms on a flag nothing sets
    st, bits = ds.dspark_read_status(ws)
    assert st == 4 and bits & ds.STATUS_TIMEOUT
    assert time.time() - t0 < 10
    # the context still works: a real op runs and matches the oracle
    cfg = SCHEDULE_CONFIGS["tiny"]
    inp = schedule_inputs(cfg)
    _, K, lengths, _ = ds.dspark_schedule(to_dev(inp["cond_accept"]), None, cfg.K_in)
    ref = oracle.schedule(inp["cond_accept"], None, cfg.K_in)
    assert int(K.item()) == ref["K"]
    np.testing.assert_array_equal(lengths.cpu().numpy(), ref["lengths"])


def test_invalid_arguments_launch_nothing(cuda_lib):
    import torch
    ds = cuda_lib
    x = torch.zeros(4, 60, dtype=torch.bfloat16, device="cuda")      # rows of 120 bytes: not TMA-able
    with pytest.raises(ds.DSparkError) as e:
        ds.dspark_draft_logits(x, torch.zeros(10, 60, dtype=torch.bfloat16, device="cuda"))
    assert e.value.status == 1
    with pytest.raises(ds.DSparkError) as e:
        ds.dspark_markov_sample(torch.zeros(1, 1, 10, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda"),
                                torch.zeros(10, 4, device="cuda"), torch.zeros(10, 4, device="cuda"),
                                torch.ones(1, device="cuda"), 0, 2 ** 33)
    assert e.value.status == 1
