"""GPU parity: verification with the draft's own Gumbel noise against the oracle.

The target's token at each position is a Gumbel-max over a whole row, computed in fp32 on the
GPU and in fp64 by the oracle: outputs must be identical for every request whose scored rows
have an oracle top-2 gap of at least NEAR_TIE_GUMBEL (the others are counted and must still be
well formed).  Drafts come from the oracle sampler (coupled with the target through the shared
noise) or from the GPU sampler itself; rows are ragged, blocks truncated, temperatures mixed
(0 scores the plain argmax and must equal greedy verification bit for bit)."""
import numpy as np
import pytest

import oracle
from tests._helpers import record_parity, to_dev

pytestmark = pytest.mark.gpu

NEAR_TIE_GUMBEL = 1e-3        # fp32 scores against fp64: rounding of t / T and of the variate


def _coupled_case(B, g, V, seed, sigma, temps):
    """Draft tokens from the oracle's Gumbel-max on draft logits d (the noise of step k), and
    target logits t = d + N(0, sigma_b^2): the closer the two, the longer the accepted runs."""
    rng = np.random.default_rng(seed)
    d = rng.standard_normal((B, g + 1, V)) * 2.0
    t = (d + rng.standard_normal((B, g + 1, V)) * np.asarray(sigma)[:, None, None]).astype(np.float32)
    T = np.asarray(temps, dtype=np.float32)
    s, off = 17, 5
    y_d, _ = oracle.target_gumbel_tokens(d[:, :g + 1], T, s, off)     # the draft's own Gumbel-max tokens
    x = y_d[:, :g].astype(np.int32)
    return t, T, x, s, off


def _check(ds, t, T, x, seed, offset, lengths=None, workspace=None):
    out, nacc = ds.dspark_verify_gumbel(to_dev(t), to_dev(T), to_dev(x), None if lengths is None else to_dev(lengths),
                                        seed, offset, workspace=workspace)
    out, nacc = out.cpu().numpy(), nacc.cpu().numpy()
    ref_out, ref_nacc, gaps = oracle.verify_gumbel(t, T, x, seed, offset, lengths, return_gaps=True)
    close = gaps < NEAR_TIE_GUMBEL
    np.testing.assert_array_equal(out[~close], ref_out[~close])
    np.testing.assert_array_equal(nacc[~close], ref_nacc[~close])
    g = x.shape[1]
    for b in np.nonzero(close)[0]:                       # near ties: well formed only
        n = nacc[b]
        assert 0 <= n <= g and np.all(out[b, :n] == x[b, :n]) and 0 <= out[b, n] < t.shape[2]
    record_parity("verify with draft noise (requests)", f"B={x.shape[0]} V={t.shape[2]}", x.shape[0], int(close.sum()))
    return ref_nacc, int(close.sum())


@pytest.mark.parametrize("B,g,V", [(6, 5, 40), (9, 4, 4097), (4, 8, 20000), (3, 3, 2048), (5, 6, 151936)])
def test_parity_coupled_drafts(cuda_lib, B, g, V):
    sigma = np.resize([0.0, 0.05, 0.3, 1.0, 3.0], B)
    temps = np.resize([1.0, 0.7, 1.3, 0.0, 2.0, 0.9], B)
    t, T, x, s, off = _coupled_case(B, g, V, 100 + V, sigma, temps)
    nacc, ties = _check(cuda_lib, t, T, x, s, off)
    assert nacc.max() >= 1                               # the coupling accepts some tokens
    print(f"B={B} V={V}: accepted {nacc.tolist()}, near ties {ties}")


def test_truncated_blocks_and_invalid_requests(cuda_lib):
    B, g, V = 8, 6, 3000
    t, T, x, s, off = _coupled_case(B, g, V, 7, np.full(B, 0.05), np.full(B, 1.0))
    lengths = np.array([0, 1, 2, 6, 5, 3, -1, 7], dtype=np.int32)   # the last two are invalid
    x[5, 1] = V                                                      # out-of-range token (tested)
    x[2, 4] = -3                                                     # out of range but past L_b
    ws = cuda_lib.Workspace(cuda_lib.OP_VERIFY_GUMBEL, B, g, V, 0)
    ref_nacc, _ = _check(cuda_lib, t, T, x, s, off, lengths, workspace=ws)
    assert np.all(ref_nacc[[5, 6, 7]] == 0)
    _, bits = cuda_lib.dspark_read_status(ws)
    assert bits & cuda_lib.STATUS_INPUT_RANGE


def test_temperature_zero_equals_greedy_verification(cuda_lib):
    rng = np.random.default_rng(3)
    B, g, V = 16, 5, 9000
    t = rng.standard_normal((B, g + 1, V)).astype(np.float32)
    am = np.argmax(t, axis=2)[:, :g]
    x = np.where(rng.random((B, g)) < 0.8, am, (am + 1) % V).astype(np.int32)
    T = np.zeros(B, dtype=np.float32)
    out, nacc = cuda_lib.dspark_verify_gumbel(to_dev(t), to_dev(T), to_dev(x), None, 1, 2)
    gout, gnacc = cuda_lib.dspark_verify_greedy(to_dev(t), to_dev(x))
    np.testing.assert_array_equal(out.cpu().numpy(), gout.cpu().numpy())
    np.testing.assert_array_equal(nacc.cpu().numpy(), gnacc.cpu().numpy())


def test_full_size_batched_draft_pipeline(cuda_lib):
    """B=64, N=16, V=151936, r=256 bf16 (the tensor-core sampler): the target scores the draft's
    own logits (base + Markov bias of the previous drafted token, the draft's temperature) and
    accepts nearly every token; four requests are checked against the oracle row by row."""
    import torch
    B, N, V, r = 64, 16, 151936, 256
    gen = torch.Generator(device="cuda")
    gen.manual_seed(11)
    L = (torch.randn(B, N, V, device="cuda", generator=gen) * 2.0).contiguous()
    w1 = torch.randn(V, r, device="cuda", generator=gen).to(torch.bfloat16)
    w2 = (torch.randn(V, r, device="cuda", generator=gen) / 16).to(torch.bfloat16)
    anchor = torch.randint(0, V, (B,), device="cuda", dtype=torch.int32, generator=gen)
    T = torch.full((B,), 0.8, device="cuda")
    s, off = 9, 2
    x = cuda_lib.dspark_markov_sample(L, anchor, w1, w2, T, s, off)
    prev = torch.cat([anchor[:, None], x[:, :-1]], dim=1).long()
    t = torch.empty(B, N + 1, V, device="cuda")
    for k in range(N):
        t[:, k] = L[:, k] + w1[prev[:, k]].float() @ w2.float().T
    t[:, N] = torch.randn(B, V, device="cuda", generator=gen)
    out, nacc = cuda_lib.dspark_verify_gumbel(t.contiguous(), T, x, None, s, off)
    nacc = nacc.cpu().numpy()
    assert nacc.mean() >= 0.9 * N, nacc
    rows = np.array([0, 21, 42, 63])
    ref_out, ref_nacc, gaps = oracle.verify_gumbel(t[rows].cpu().numpy(), np.full(4, 0.8), x[rows].cpu().numpy(),
                                                   s, off, return_gaps=True, req_ids=rows)
    ok = gaps >= NEAR_TIE_GUMBEL
    np.testing.assert_array_equal(out.cpu().numpy()[rows][ok], ref_out[ok])
    np.testing.assert_array_equal(nacc[rows][ok], ref_nacc[ok])


def test_sampler_pipeline_accepts_its_own_logits(cuda_lib):
    """The GPU Markov sampler drafts; a target whose rows are the draft's own scaled logits
    (base + Markov bias of the previous drafted token, the draft's temperature) accepts nearly
    every token (fp32 rounding of the two evaluations may split a near tie)."""
    import torch
    rng = np.random.default_rng(5)
    B, N, V, r = 16, 8, 30000, 64
    L = (rng.standard_normal((B, N, V)) * 2).astype(np.float32)
    w1 = rng.standard_normal((V, r)).astype(np.float32)
    w2 = (rng.standard_normal((V, r)) / 8).astype(np.float32)
    anchor = rng.integers(0, V, B).astype(np.int32)
    T = np.full(B, 0.8, np.float32)
    s, off = 4, 6
    x = cuda_lib.dspark_markov_sample(to_dev(L), to_dev(anchor), to_dev(w1), to_dev(w2), to_dev(T), s, off)
    xh = x.cpu().numpy()
    prev = np.concatenate([anchor[:, None], xh[:, :-1]], axis=1)
    t = np.empty((B, N + 1, V), np.float32)
    for k in range(N):
        t[:, k] = L[:, k] + oracle.markov_bias(prev[:, k], w1, w2)
    t[:, N] = rng.standard_normal((B, V))
    out, nacc = cuda_lib.dspark_verify_gumbel(to_dev(t), to_dev(T), x, None, s, off)
    nacc = nacc.cpu().numpy()
    assert nacc.mean() >= 0.9 * N, nacc
    np.testing.assert_array_equal(out.cpu().numpy()[:, :N][nacc == N], xh[nacc == N])
