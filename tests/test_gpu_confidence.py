"""GPU parity: calibrated confidence head against the oracle (fp32 on the GPU, fp64 in the
oracle; |difference| <= 2e-5, from fp32 sums of up to 4096 terms of size O(1/sqrt(H))), and the
head feeding the scheduler."""
import numpy as np
import pytest

import oracle
from tests._helpers import to_dev
from workloads import DRAFT_CONFIGS, draft_inputs, normal_rows, to_bf16_values

pytestmark = pytest.mark.gpu
TOL = 2e-5


def _head(H, r, N, seed):
    rng = np.random.default_rng(seed)
    w_h = (rng.standard_normal(H) / np.sqrt(H)).astype(np.float32)
    w_e = (rng.standard_normal(r) / np.sqrt(r) * 0.3).astype(np.float32)
    tau = rng.uniform(0.7, 1.6, N).astype(np.float32)
    return w_h, w_e, float(np.float32(rng.standard_normal() * 0.5 + 1.0)), tau


@pytest.mark.parametrize("name", ["tiny", "qwen3_8b_single", "batched_draft"])
def test_workload_shapes(cuda_lib, name):
    """The draft workloads' shapes and dtypes (hidden rows RMS-normalised, w1 as the Markov head's)."""
    cfg = DRAFT_CONFIGS[name]
    B, N, H, V, r = cfg.B, cfg.N, cfg.H, cfg.V, cfg.r
    hidden = normal_rows(B * N, H, 1.0, cfg.data_seed, "hidden")
    hidden = (hidden / np.sqrt(np.mean(hidden.astype(np.float64) ** 2, axis=1, keepdims=True))).astype(np.float32)
    w1 = normal_rows(V, r, 1.0, cfg.data_seed, "w1")
    import torch
    if cfg.dtype == "bf16":
        th, hidden = to_bf16_values(hidden)
        tw1, w1 = to_bf16_values(w1)
    else:
        th, tw1 = torch.from_numpy(hidden), torch.from_numpy(w1)
    rng = np.random.default_rng(1)
    x = rng.integers(0, V, (B, N)).astype(np.int32)
    a = rng.integers(0, V, B).astype(np.int32)
    w_h, w_e, beta, tau = _head(H, r, N, 2)
    conf = cuda_lib.dspark_confidence(th.cuda(), tw1.cuda(), to_dev(a), to_dev(x), to_dev(w_h), to_dev(w_e), beta,
                                      to_dev(tau))
    ref = oracle.confidence(hidden, w1, a, x, w_h, w_e, beta, tau)
    np.testing.assert_allclose(conf.cpu().numpy(), ref, rtol=0, atol=TOL)


@pytest.mark.parametrize("H,r,dt", [(1, 1, "f32"), (7, 3, "f32"), (100, 24, "bf16"), (4099, 65, "bf16")])
def test_ragged_sizes_and_dtypes(cuda_lib, H, r, dt):
    B, N, V = 5, 7, 300
    hidden = normal_rows(B * N, H, 1.0, H, "hidden")
    w1 = normal_rows(V, r, 1.0, H, "w1")
    import torch
    if dt == "bf16":
        th, hidden = to_bf16_values(hidden)
        tw1, w1 = to_bf16_values(w1)
    else:
        th, tw1 = torch.from_numpy(hidden), torch.from_numpy(w1)
    rng = np.random.default_rng(H)
    x = rng.integers(0, V, (B, N)).astype(np.int32)
    a = rng.integers(0, V, B).astype(np.int32)
    w_h, w_e, beta, tau = _head(H, r, N, H + 1)
    conf = cuda_lib.dspark_confidence(th.cuda(), tw1.cuda(), to_dev(a), to_dev(x), to_dev(w_h), to_dev(w_e), beta,
                                      to_dev(tau))
    np.testing.assert_allclose(conf.cpu().numpy(), oracle.confidence(hidden, w1, a, x, w_h, w_e, beta, tau),
                               rtol=0, atol=TOL)


def test_bad_previous_token_and_temperature_set_flags(cuda_lib):
    B, N, H, V, r = 2, 3, 16, 50, 4
    import torch
    hidden = torch.randn(B * N, H, device="cuda")
    w1 = torch.randn(V, r, device="cuda")
    x = torch.tensor([[1, 2, 3], [4, V + 7, 5]], dtype=torch.int32, device="cuda")
    a = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    tau = torch.tensor([1.0, 0.0, 1.0], device="cuda")
    ws = cuda_lib.Workspace(cuda_lib.OP_CONFIDENCE, B, N, V, r)
    conf = cuda_lib.dspark_confidence(hidden, w1, a, x, torch.zeros(H, device="cuda"), torch.zeros(r, device="cuda"),
                                      0.0, tau, workspace=ws)
    st, bits = cuda_lib.dspark_read_status(ws)
    assert bits & cuda_lib.STATUS_INPUT_RANGE and bits & cuda_lib.STATUS_NUMERIC
    c = conf.cpu().numpy()
    assert np.all(c[:, 1] == 0.0) and np.allclose(c[:, [0, 2]], 0.5)


def test_head_feeds_the_scheduler(cuda_lib):
    """conf from the head is the scheduler's cond_accept: the admission equals the oracle's on
    the oracle's own confidences where those round to the same float32 values."""
    cfg = DRAFT_CONFIGS["tiny"]
    inp = draft_inputs(cfg)
    B, N, H, V, r = 4, cfg.N, cfg.H, cfg.V, cfg.r
    rng = np.random.default_rng(3)
    hidden = normal_rows(B * N, H, 1.0, 3, "hidden")
    x = rng.integers(0, V, (B, N)).astype(np.int32)
    a = rng.integers(0, V, B).astype(np.int32)
    w_h, w_e, beta, tau = _head(H, r, N, 4)
    conf = cuda_lib.dspark_confidence(to_dev(hidden), to_dev(inp["w1_f32"]), to_dev(a), to_dev(x), to_dev(w_h),
                                      to_dev(w_e), beta, to_dev(tau))
    from workloads import sps_table
    sps = sps_table(B * N)
    surv, K, lengths, sel = cuda_lib.dspark_schedule(conf, to_dev(sps), -1)
    ref = oracle.schedule(conf.cpu().numpy(), sps, -1)          # same float32 confidences on both sides
    assert int(K.item()) == ref["K"]
    np.testing.assert_array_equal(lengths.cpu().numpy(), ref["lengths"])
