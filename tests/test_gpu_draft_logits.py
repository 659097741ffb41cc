"""GPU parity: base logits of the draft LM head (tcgen05 GEMM) against the fp64 oracle.

Tolerance: max |gpu - oracle| <= 2e-2 on every compared element (bf16 inputs are
multiplied exactly and summed in fp32; fp32 inputs run as tf32).
"""
import numpy as np
import pytest

import oracle
from tests._helpers import LOGIT_TOL, to_dev
from workloads import DRAFT_CONFIGS, draft_inputs, normal_rows, to_bf16_values

pytestmark = pytest.mark.gpu


def _run(ds, X, W):
    import torch
    L = ds.dspark_draft_logits(X, W)
    torch.cuda.synchronize()
    return L.cpu().numpy()


def test_tiny_fp32_tf32_full(cuda_lib):
    cfg = DRAFT_CONFIGS["tiny"]
    inp = draft_inputs(cfg)
    got = _run(cuda_lib, to_dev(inp["hidden"]), to_dev(inp["lm_head"]))
    ref = oracle.draft_logits(inp["hidden_f32"], inp["lm_head_f32"])
    assert np.abs(got - ref).max() <= LOGIT_TOL


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("M,H,V", [(1, 64, 1), (3, 136, 100), (8, 256, 1000), (17, 200, 4097),
                                   (100, 64, 333), (129, 128, 520), (256, 64, 300),
                                   (300, 192, 777), (513, 72, 1031), (384, 128, 129),
                                   (640, 256, 2000), (1024, 64, 256), (5, 1096, 3000), (24, 1352, 2100),
                                   (300, 128, 11900), (1024, 64, 5000), (520, 96, 13000)])
def test_ragged_shapes(cuda_lib, dtype, M, H, V):
    """Several tiles with ragged tails in M, V and K, in both tile shapes (swap for M <= 256; above,
    CTA-pair 256 x 256 tiles for bf16, including pairs whose second half lies wholly past M or V).
    The decode tiles put four (M <= 16) or two (M <= 32) K slices in a stage: H = 1096 and 1352
    wrap their rings several times per tile and end on a stage with fewer slices.  94, 80 and 153
    pair tiles take the persistent pairs more than one round, ending on a partial round, with V
    ending 124, 136 and 200 entries into the last tile."""
    if dtype == "f32" and H % 4:
        pytest.skip("fp32 rows must be 16-byte multiples")
    X = normal_rows(M, H, 1.0, 77, "hidden")
    W = normal_rows(V, H, 1.0 / np.sqrt(H), 77, "lm_head")
    if dtype == "bf16":
        tX, X = to_bf16_values(X)
        tW, W = to_bf16_values(W)
    else:
        import torch
        tX, tW = torch.from_numpy(X), torch.from_numpy(W)
    got = _run(cuda_lib, to_dev(tX), to_dev(tW))
    ref = oracle.draft_logits(X, W)
    assert got.shape == (M, V)
    assert np.abs(got - ref).max() <= LOGIT_TOL


def test_qwen3_8b_single_request_full(cuda_lib):
    """B=1, N=8, H=4096, V=151936, bf16: every logit compared."""
    cfg = DRAFT_CONFIGS["qwen3_8b_single"]
    inp = draft_inputs(cfg)
    got = _run(cuda_lib, to_dev(inp["hidden"]), to_dev(inp["lm_head"]))
    ref = oracle.draft_logits(inp["hidden_f32"], inp["lm_head_f32"])
    err = np.abs(got - ref).max()
    print(f"qwen3_8b_single draft_logits max abs err {err:.3e}")
    assert err <= LOGIT_TOL


def test_batched_draft_full_size_sampled(cuda_lib):
    """B=64, N=16 (M=1024), bf16: 24 sampled rows in full plus 64 sampled columns of every row."""
    cfg = DRAFT_CONFIGS["batched_draft"]
    inp = draft_inputs(cfg)
    got = _run(cuda_lib, to_dev(inp["hidden"]), to_dev(inp["lm_head"]))
    rng = np.random.default_rng(3)
    M = cfg.B * cfg.N
    rows = np.unique(np.concatenate([[0, M - 1, 127, 128], rng.choice(M, 20, replace=False)]))
    ref_rows = oracle.draft_logits(inp["hidden_f32"][rows], inp["lm_head_f32"])
    assert np.abs(got[rows] - ref_rows).max() <= LOGIT_TOL
    cols = np.unique(np.concatenate([[0, cfg.V - 1, 255, 256], rng.choice(cfg.V, 60, replace=False)]))
    ref_cols = oracle.draft_logits(inp["hidden_f32"], inp["lm_head_f32"][cols])
    assert np.abs(got[:, cols] - ref_cols).max() <= LOGIT_TOL


def test_identity_lm_head_returns_hidden(cuda_lib):
    """H = V and lm_head = I: logits = hidden exactly (bf16 values, fp32 sums of one term)."""
    import torch
    H = 256
    X = normal_rows(5, H, 1.0, 5, "hidden")
    tX, X = to_bf16_values(X)
    tW = torch.eye(H, dtype=torch.bfloat16)
    got = _run(cuda_lib, to_dev(tX), to_dev(tW))
    np.testing.assert_array_equal(got, X)
