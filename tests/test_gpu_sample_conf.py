"""GPU parity: the Markov sampler with the calibrated confidence head evaluated inside it.

The tokens must be exactly those of dspark_markov_sample with the same inputs and Philox stream
(the head only reads what the sampler holds), and match the oracle under the teacher-forced
near-tie rule.  The confidences must be within 2e-5 of the oracle's confidence head evaluated on
the tokens the GPU drew ("Speculative decoding: from zero to DSpark" §6: the head sees the
embedding of the previous draft token, so the draft's own tokens are the ones that count), on
both sampler paths and at every draft workload.  Fed to dspark_schedule, they give the oracle's
admission of the same float32 values bit for bit.
"""
import numpy as np
import pytest

import oracle
from tests._helpers import check_markov_parity, to_dev
from workloads import DRAFT_CONFIGS, DraftConfig, draft_inputs, markov_logits, normal_rows, sps_table, to_bf16_values

pytestmark = pytest.mark.gpu
TOL = 2e-5          # fp32 sums of up to 4096 terms of size O(1/sqrt(H)) against fp64


def _head(H, r, N, seed):
    rng = np.random.default_rng(seed)
    w_h = (rng.standard_normal(H) / np.sqrt(H)).astype(np.float32)
    w_e = (rng.standard_normal(r) / np.sqrt(r) * 0.3).astype(np.float32)
    tau = rng.uniform(0.7, 1.6, N).astype(np.float32)
    return w_h, w_e, float(np.float32(rng.standard_normal() * 0.5 + 1.0)), tau


def _run(ds, L, anchor, tw1, tw2, T, seed, offset, th, head):
    w_h, w_e, beta, tau = head
    B, N, V = L.shape
    ws = ds.Workspace(ds.OP_MARKOV_SAMPLE, B, N, V, tw1.shape[1])
    args = (to_dev(L), to_dev(anchor), tw1.cuda(), tw2.cuda(), to_dev(T), seed, offset)
    tok, conf = ds.dspark_markov_sample_conf(*args, th.cuda(), to_dev(w_h), to_dev(w_e), beta, to_dev(tau),
                                             workspace=ws)
    st, bits = ds.dspark_read_status(ws)
    plain = ds.dspark_markov_sample(*args).cpu().numpy()
    return tok.cpu().numpy(), conf.cpu().numpy(), st, bits, plain


@pytest.mark.parametrize("name", ["tiny", "qwen3_8b_single", "batched_draft"])
def test_fused_head_at_the_draft_workloads(cuda_lib, name):
    cfg = DRAFT_CONFIGS[name]
    inp = draft_inputs(cfg)
    L = markov_logits(cfg)
    T = np.full(cfg.B, cfg.temperatures[-1], np.float32)
    head = _head(cfg.H, cfg.r, cfg.N, 11)
    tok, conf, st, bits, plain = _run(cuda_lib, L, inp["anchor"], inp["w1"], inp["w2"], T, 5, 2, inp["hidden"], head)
    assert st == 0, bits
    np.testing.assert_array_equal(tok, plain)
    check_markov_parity(tok, L, inp["anchor"], inp["w1_f32"], inp["w2_f32"], T, 5, 2, label=f"fused head {name}")
    ref = oracle.confidence(inp["hidden_f32"], inp["w1_f32"], inp["anchor"], tok, *head)
    np.testing.assert_allclose(conf, ref, rtol=0, atol=TOL)


@pytest.mark.parametrize("B,N,V,r,H,dt,T", [(20, 3, 20004, 128, 100, "bf16", 0.9), (3, 4, 5000, 24, 7, "f32", 1.1),
                                              (33, 2, 65536, 256, 4099, "bf16", 0.0), (1, 6, 70001, 64, 256, "bf16", 1.0)])
def test_ragged_shapes_both_paths(cuda_lib, B, N, V, r, H, dt, T):
    """Padded request chunks on the tensor path (B = 20, 33), the CUDA-core path (fp32 head,
    B = 3), greedy requests, the single-request decode path (bf16, r = 64), ragged H."""
    cfg = DraftConfig("conf", B=B, N=N, H=H, V=V, r=r, dtype=dt, temperatures=(T,), data_seed=B + V)
    L = markov_logits(cfg, scale=1.5)
    w1 = normal_rows(V, r, 1.0, B + V, "w1")
    w2 = normal_rows(V, r, 1.0 / np.sqrt(r), B + V, "w2")
    hidden = normal_rows(B * N, H, 1.0, B + V, "hidden")
    import torch
    if dt == "bf16":
        tw1, w1 = to_bf16_values(w1)
        tw2, w2 = to_bf16_values(w2)
        th, hidden = to_bf16_values(hidden)
    else:
        tw1, tw2, th = torch.from_numpy(w1), torch.from_numpy(w2), torch.from_numpy(hidden)
    anchor = np.random.default_rng(B).integers(0, V, B).astype(np.int32)
    Ts = np.full(B, T, np.float32)
    head = _head(H, r, N, B * 3 + 1)
    tok, conf, st, bits, plain = _run(cuda_lib, L, anchor, tw1, tw2, Ts, 7, 1, th, head)
    assert st == 0, bits
    np.testing.assert_array_equal(tok, plain)
    check_markov_parity(tok, L, anchor, w1, w2, Ts, 7, 1, label=f"fused head B={B} V={V} r={r} {dt}")
    np.testing.assert_allclose(conf, oracle.confidence(hidden, w1, anchor, tok, *head), rtol=0, atol=TOL)


def test_bad_calibration_temperature_gives_zero_and_flag(cuda_lib):
    cfg = DRAFT_CONFIGS["tiny"]
    inp = draft_inputs(cfg)
    L = markov_logits(cfg)
    w_h, w_e, beta, tau = _head(cfg.H, cfg.r, cfg.N, 3)
    tau[2] = 0.0
    tok, conf, st, bits, _ = _run(cuda_lib, L, inp["anchor"], inp["w1"], inp["w2"], np.ones(1, np.float32), 0, 0,
                                  inp["hidden"], (w_h, w_e, beta, tau))
    assert bits & cuda_lib.STATUS_NUMERIC
    assert conf[0, 2] == 0.0 and np.all(conf[0, [0, 1, 3]] > 0)


def test_fused_head_feeds_the_scheduler(cuda_lib):
    """The batched draft step's confidences are the scheduler's cond_accept: the admission
    equals the oracle's on the same float32 values, bit for bit."""
    cfg = DRAFT_CONFIGS["batched_draft"]
    inp = draft_inputs(cfg)
    L = markov_logits(cfg)
    T = np.full(cfg.B, 0.8, np.float32)
    head = _head(cfg.H, cfg.r, cfg.N, 9)
    tok, conf, st, _, _ = _run(cuda_lib, L, inp["anchor"], inp["w1"], inp["w2"], T, 0, 0, inp["hidden"], head)
    assert st == 0
    sps = sps_table(cfg.B * cfg.N)
    surv, K, lengths, sel = cuda_lib.dspark_schedule(to_dev(conf), to_dev(sps), -1)
    ref = oracle.schedule(conf, sps, -1)
    assert int(K.item()) == ref["K"]
    np.testing.assert_array_equal(lengths.cpu().numpy(), ref["lengths"])
    np.testing.assert_array_equal(sel.cpu().numpy(), ref["selected"])
    np.testing.assert_array_equal(surv.cpu().numpy(), ref["survival"])
