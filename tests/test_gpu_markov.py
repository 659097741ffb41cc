"""GPU parity: sequential Markov-biased Gumbel-max sampling against the oracle.

Every position of every request is compared: the oracle runs each step on the
GPU's own previous token (teacher forcing), and a token may differ only where
the oracle's top-2 gap of perturbed values is below 5e-2.  Such near-tie
divergences are counted, bounded and recorded (printed at the end of the run).
Inputs are the same seeded synthetic tensors on both sides, with the shared
Philox stream.
"""
import numpy as np
import pytest

import oracle
from tests._helpers import check_markov_parity, to_dev
from workloads import (DRAFT_CONFIGS, DraftConfig, draft_inputs, draft_inputs_markov, markov_logits,
                       normal_rows, to_bf16_values)

pytestmark = pytest.mark.gpu


def _gpu(ds, L, anchor, w1, w2, T, seed, offset, lse=False):
    import torch
    B, N, _ = L.shape
    lse_t = torch.empty(B, N, dtype=torch.float32, device="cuda") if lse else None
    ws = ds.Workspace(ds.OP_MARKOV_SAMPLE, B, N, L.shape[2], w1.shape[1])
    tok = ds.dspark_markov_sample(to_dev(L), to_dev(anchor), to_dev(w1), to_dev(w2), to_dev(T),
                                  seed, offset, lse=lse_t, workspace=ws)
    st, bits = ds.dspark_read_status(ws)
    return tok.cpu().numpy(), (lse_t.cpu().numpy() if lse else None), st, bits


def test_tiny_fp32(cuda_lib):
    cfg = DRAFT_CONFIGS["tiny"]
    inp = draft_inputs(cfg)
    L = markov_logits(cfg)
    T = np.ones(cfg.B, np.float32)
    tok, lse, st, _ = _gpu(cuda_lib, L, inp["anchor"], inp["w1"], inp["w2"], T, 0, 0, lse=True)
    assert st == 0
    _, _, rlse = check_markov_parity(tok, L, inp["anchor"], inp["w1_f32"], inp["w2_f32"], T, 0, 0, label="tiny")
    np.testing.assert_allclose(lse, rlse, rtol=0, atol=1e-3)


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_qwen3_8b_single_request(cuda_lib, T):
    """B=1, N=8, V=151936, r=64, bf16 weights; greedy and T=1."""
    cfg = DRAFT_CONFIGS["qwen3_8b_single"]
    inp = draft_inputs(cfg)
    L = markov_logits(cfg)
    Ts = np.full(cfg.B, T, np.float32)
    for seed, offset in ((0, 0), (12345, 7)):
        tok, _, st, _ = _gpu(cuda_lib, L, inp["anchor"], inp["w1"], inp["w2"], Ts, seed, offset)
        assert st == 0
        check_markov_parity(tok, L, inp["anchor"], inp["w1_f32"], inp["w2_f32"], Ts, seed, offset,
                            label=f"qwen3_8b_single T={T} seed={seed}")


def test_batched_draft_all_requests(cuda_lib):
    """B=64, N=16, V=151936, r=256, T=0.8, Zipf-ranked logits and spiked w1: all 64 requests,
    every position, and the lse output at every position (on the GPU's own prefix)."""
    cfg = DRAFT_CONFIGS["batched_draft"]
    inp = draft_inputs_markov(cfg)
    L = markov_logits(cfg)
    T = np.full(cfg.B, 0.8, np.float32)
    tok, lse, st, _ = _gpu(cuda_lib, L, inp["anchor"], inp["w1"], inp["w2"], T, 0, 0, lse=True)
    assert st == 0
    n, _, rlse = check_markov_parity(tok, L, inp["anchor"], inp["w1_f32"], inp["w2_f32"], T, 0, 0,
                                     label="batched_draft")
    assert n == cfg.B * cfg.N
    np.testing.assert_allclose(lse, rlse, rtol=0, atol=2e-3)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,N,V,r,T", [(1, 1, 2, 1, 1.0), (3, 5, 1001, 5, 0.7), (2, 4, 4097, 16, 0.0),
                                       (5, 3, 40000, 64, 1.3), (16, 2, 3000, 256, 0.9),
                                       (1, 6, 2000, 64, 1.0), (1, 5, 70001, 64, 0.8), (1, 3, 9000, 64, 0.0)])
def test_ragged_and_edge_shapes(cuda_lib, dtype, B, N, V, r, T):
    """Includes single requests at r = 64 (bf16: the bias on the tensor cores) with slices of
    a few hundred entries and a ragged last slice."""
    cfg = DraftConfig("edge", B=B, N=N, H=8, V=V, r=r, dtype=dtype, temperatures=(T,), data_seed=91)
    L = markov_logits(cfg, scale=2.0)
    w1 = normal_rows(V, r, 1.0, 91, "w1")
    w2 = normal_rows(V, r, 1.0 / np.sqrt(r), 91, "w2")
    if dtype == "bf16":
        tw1, w1 = to_bf16_values(w1)
        tw2, w2 = to_bf16_values(w2)
    else:
        import torch
        tw1, tw2 = torch.from_numpy(w1), torch.from_numpy(w2)
    anchor = np.random.default_rng(B * 7 + V).integers(0, V, B).astype(np.int32)
    Ts = np.full(B, T, np.float32)
    tok, _, st, _ = _gpu(cuda_lib, L, anchor, tw1, tw2, Ts, 3, 1)
    assert st == 0
    check_markov_parity(tok, L, anchor, w1, w2, Ts, 3, 1, label=f"edge {dtype} B={B} N={N} V={V} r={r} T={T}")


def test_zero_markov_head_is_independent_gumbel_max(cuda_lib):
    """w1 = 0: every position is the Gumbel-max of its own base logits (same Philox stream)."""
    import torch
    B, N, V, r = 4, 6, 5000, 8
    cfg = DraftConfig("z", B=B, N=N, H=8, V=V, r=r, dtype="f32", temperatures=(1.0,), data_seed=5)
    L = markov_logits(cfg)
    w1 = np.zeros((V, r), np.float32)
    w2 = normal_rows(V, r, 1.0, 5, "w2")
    T = np.ones(B, np.float32)
    tok, _, st, _ = _gpu(cuda_lib, L, np.zeros(B, np.int32), torch.from_numpy(w1), torch.from_numpy(w2),
                         T, 11, 0)
    from oracle.philox import draft_gumbel
    for i in range(N):
        y = L[:, i, :].astype(np.float64) + draft_gumbel(11, 0, np.arange(B), i, V)
        ref = np.argmax(y, axis=1)
        srt = np.sort(y, axis=1)
        gap = srt[:, -1] - srt[:, -2]
        ok = (tok[:, i] == ref) | (gap < 5e-2)
        assert ok.all()


def test_deterministic_and_offset_changes_stream(cuda_lib):
    cfg = DRAFT_CONFIGS["tiny"]
    inp = draft_inputs(cfg)
    L = markov_logits(cfg, scale=0.3)
    T = np.ones(cfg.B, np.float32)
    a, _, _, _ = _gpu(cuda_lib, L, inp["anchor"], inp["w1"], inp["w2"], T, 1, 0)
    b, _, _, _ = _gpu(cuda_lib, L, inp["anchor"], inp["w1"], inp["w2"], T, 1, 0)
    c, _, _, _ = _gpu(cuda_lib, L, inp["anchor"], inp["w1"], inp["w2"], T, 1, 1)
    np.testing.assert_array_equal(a, b)
    assert not np.array_equal(a, c)


def test_anchor_out_of_range_sets_status(cuda_lib):
    cfg = DRAFT_CONFIGS["tiny"]
    inp = draft_inputs(cfg)
    L = markov_logits(cfg)
    _, _, st, bits = _gpu(cuda_lib, L, np.array([cfg.V + 5], np.int32), inp["w1"], inp["w2"],
                          np.ones(1, np.float32), 0, 0)
    assert bits & cuda_lib.STATUS_INPUT_RANGE and st == 6


@pytest.mark.parametrize("V", [1000, 151936])
def test_step_without_finite_logits_sets_numeric_and_spares_other_requests(cuda_lib, V):
    """One request's base logits are NaN at one step: that step has no candidate (token 0 and the
    NUMERIC bit); the other request still matches the oracle."""
    B, N, r = 2, 3, 64
    cfg = DraftConfig("nan", B=B, N=N, H=8, V=V, r=r, dtype="f32", temperatures=(1.0,), data_seed=3)
    L = markov_logits(cfg)
    L[1, 1, :] = np.nan
    w1 = normal_rows(V, r, 1.0, 3, "w1")
    w2 = normal_rows(V, r, 1.0 / np.sqrt(r), 3, "w2")
    import torch
    anchor = np.array([5, 9], np.int32)
    T = np.ones(B, np.float32)
    tok, _, st, bits = _gpu(cuda_lib, L, anchor, torch.from_numpy(w1), torch.from_numpy(w2), T, 4, 0)
    assert bits & cuda_lib.STATUS_NUMERIC
    assert tok[1, 1] == 0
    check_markov_parity(tok[:1], L[:1], anchor[:1], w1, w2, T[:1], 4, 0, label=f"nan-step V={V}")


def test_single_request_bf16_step_without_finite_logits(cuda_lib):
    """One request, bf16 head at r = 64 (the tensor-core bias): a step whose base logits are all
    NaN has no candidate (token 0, NUMERIC bit); the step before it matches the oracle and the
    call completes."""
    B, N, V, r = 1, 4, 20000, 64
    cfg = DraftConfig("nan1", B=B, N=N, H=8, V=V, r=r, dtype="bf16", temperatures=(1.0,), data_seed=8)
    L = markov_logits(cfg)
    L[0, 2, :] = np.nan
    tw1, w1 = to_bf16_values(normal_rows(V, r, 1.0, 8, "w1"))
    tw2, w2 = to_bf16_values(normal_rows(V, r, 1.0 / np.sqrt(r), 8, "w2"))
    anchor = np.array([17], np.int32)
    T = np.ones(B, np.float32)
    tok, _, st, bits = _gpu(cuda_lib, L, anchor, tw1, tw2, T, 6, 0)
    assert bits & cuda_lib.STATUS_NUMERIC and not bits & cuda_lib.STATUS_TIMEOUT
    assert tok[0, 2] == 0
    check_markov_parity(tok[:, :2], L[:, :2], anchor, w1, w2, T, 6, 0, label="nan-step bf16 r=64")
