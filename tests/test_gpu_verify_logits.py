"""GPU parity: verification from logits (draft distribution recomputed) against the oracle.

The device evaluates p_t and p_d in fp32 from logits, normalisers and the Markov bias; the
oracle in fp64.  A decision may then differ only where it sits within rounding of its
boundary, so each request is compared under this rule:
  * if every acceptance test the oracle made has a relative margin |u p_d - p_t| / p_t of at
    least ACCEPT_MARGIN, num_accepted and the accepted prefix must be identical;
  * if in addition the oracle's draw has a top-2 gap of perturbed values of at least the
    gap tolerance, the correction / bonus token must be identical too.
Requests inside a margin are counted (and must still be well formed); their share is bounded.
The draft's log-sum-exp input is the oracle's (float32), standing for the sampler's output.
"""
import numpy as np
import pytest

import oracle
from tests._helpers import record_parity, to_dev
from workloads import VERIFY_LOGITS_CONFIGS, VerifyLogitsConfig, verify_logits_inputs

pytestmark = pytest.mark.gpu

ACCEPT_MARGIN = 1e-4      # relative; fp32 p_t(x), p_d(x) are within ~1e-5 of exact
GAP = 1e-3                # perturbed values carry ~1e-5 of fp32 rounding (logs, exps, the bias dot)


def _torch_inputs(inp, lse):
    import torch
    d = {k: to_dev(inp[k]) for k in ("target_logits", "base_logits", "anchor", "T_t", "T_d", "draft_tokens")}
    d["w1"] = inp["w1"].cuda()
    d["w2"] = inp["w2"].cuda()
    d["lse"] = to_dev(lse.astype(np.float32))
    d["lengths"] = None if inp["lengths"] is None else to_dev(inp["lengths"])
    return d


def _run(ds, d, seed, offset, workspace=None):
    return ds.dspark_verify_logits(d["target_logits"], d["T_t"], d["base_logits"], d["anchor"], d["w1"], d["w2"],
                                   d["T_d"], d["lse"], d["draft_tokens"], d["lengths"], seed, offset,
                                   workspace=workspace)


def _oracle(inp, seed, offset, rows=None):
    rows = np.arange(inp["draft_tokens"].shape[0]) if rows is None else np.asarray(rows)
    lengths = None if inp["lengths"] is None else inp["lengths"][rows]
    return oracle.verify_from_logits(inp["target_logits"][rows], inp["T_t"][rows], inp["base_logits"][rows],
                                     inp["anchor"][rows], inp["w1_f32"], inp["w2_f32"], inp["T_d"][rows],
                                     inp["draft_tokens"][rows], lengths, seed, offset, req_ids=rows)


def _compare(out, nacc, x, ref, V, gap_tol, rows=None):
    """Returns the number of requests inside a margin; raises on a real mismatch."""
    ref_out, ref_nacc, acc_margin, gap = ref
    rows = np.arange(len(ref_nacc)) if rows is None else np.asarray(rows)
    near = 0
    for i, b in enumerate(rows):
        n = int(nacc[b])
        assert 0 <= n <= x.shape[1]
        np.testing.assert_array_equal(out[b, :n], x[b, :n])
        assert 0 <= out[b, n] < V and np.all(out[b, n + 1:] == -1), f"request {b} malformed: {out[b]}"
        if acc_margin[i] < ACCEPT_MARGIN:
            near += 1
            continue
        assert n == ref_nacc[i], f"request {b}: gpu accepted {n}, oracle {ref_nacc[i]} (margin {acc_margin[i]:.3g})"
        if gap[i] < gap_tol:
            near += 1
            continue
        assert out[b, n] == ref_out[i, n], (
            f"request {b}: gpu token {out[b, n]}, oracle {ref_out[i, n]} (gap {gap[i]:.3g})")
    record_parity("verify from logits (requests)", f"B={len(rows)} V={V}", len(rows), near)
    return near


def _small_cfg(dtype, V, seed, temps=(0.0, 0.7, 1.0), r=64, B=37, gamma=4):
    return VerifyLogitsConfig(f"small_{dtype}_{V}", B=B, gamma=gamma, V=V, r=r, dtype=dtype, target_std=2.0,
                              draft_sigmas=(0.3, 1.0, 3.0), draft_temps=temps, target_temp=0.8,
                              data_seed=seed, ragged_lengths=True)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [2, 4096, 5001, 20003])
def test_parity_small(cuda_lib, dtype, V):
    """Ragged vocabularies (scalar tails, several 2048-entry chunks), ragged lengths, greedy and
    sampled drafts mixed in one batch, both weight dtypes."""
    cfg = _small_cfg(dtype, V, 100 + V)
    inp = verify_logits_inputs(cfg)
    lse = oracle.draft_lse(inp["base_logits"], inp["anchor"], inp["w1_f32"], inp["w2_f32"], inp["T_d"],
                           inp["draft_tokens"])
    out, nacc = _run(cuda_lib, _torch_inputs(inp, lse), 11, 3)
    ref = _oracle(inp, 11, 3)
    near = _compare(out.cpu().numpy(), nacc.cpu().numpy(), inp["draft_tokens"], ref, V,
                    GAP)
    assert near <= max(2, cfg.B // 10)
    assert ref[1].max() >= 1                      # some blocks accept tokens


def test_full_size_sampled(cuda_lib):
    """B=256, gamma=8, V=151936, r=256 bf16: the whole batch on the GPU, 12 requests (all three
    draft-noise levels) by the oracle."""
    cfg = VERIFY_LOGITS_CONFIGS["verify"]
    inp = verify_logits_inputs(cfg)
    lse = oracle.draft_lse(inp["base_logits"], inp["anchor"], inp["w1_f32"], inp["w2_f32"], inp["T_d"],
                           inp["draft_tokens"])
    out, nacc = _run(cuda_lib, _torch_inputs(inp, lse), cfg.verify_seed, 0)
    out, nacc = out.cpu().numpy(), nacc.cpu().numpy()
    rows = np.concatenate([np.flatnonzero(inp["sigma"] == s)[:4] for s in cfg.draft_sigmas])
    ref = _oracle(inp, cfg.verify_seed, 0, rows)
    near = _compare(out, nacc, inp["draft_tokens"], ref, cfg.V, GAP, rows)
    assert near <= 2
    # every request well formed
    for b in range(cfg.B):
        n = nacc[b]
        assert 0 <= n <= cfg.gamma and np.all(out[b, :n] == inp["draft_tokens"][b, :n])
        assert 0 <= out[b, n] < cfg.V and np.all(out[b, n + 1:] == -1)


@pytest.mark.parametrize("T_d", [1.3, 0.0])
def test_lossless_law(cuda_lib, T_d):
    """40000 requests sharing one set of rows, draft tokens drawn by the oracle's sampler: the first
    emitted token follows target row 0, and given an accepted first token the second follows row
    1 (which needs the position-1 draft distribution conditioned on x_0).  A subset is also
    compared with the oracle request by request."""
    from scipy import stats
    import torch
    rng = np.random.default_rng(21)
    B, g, V, r = 40000, 2, 8, 8
    t = (rng.standard_normal((g + 1, V)) * 1.5).astype(np.float32)
    Lr = (t[:g] / 0.8 if T_d == 0 else rng.standard_normal((g, V))).astype(np.float32)
    w1 = rng.standard_normal((V, r)).astype(np.float32)
    w2 = (rng.standard_normal((V, r)) * (0.3 if T_d == 0 else 1.0)).astype(np.float32)
    tb = np.ascontiguousarray(np.broadcast_to(t, (B, g + 1, V)))
    Lb = np.ascontiguousarray(np.broadcast_to(Lr, (B, g, V)))
    anchor = np.full(B, 3, np.int32)
    Tt, Td = np.full(B, 0.8, np.float32), np.full(B, T_d, np.float32)
    x, _, _ = oracle.markov_sample(Lb, anchor, w1, w2, Td, 4, 0)
    x = x.astype(np.int32)
    lse = oracle.draft_lse(Lb, anchor, w1, w2, Td, x)
    inp = {"target_logits": tb, "base_logits": Lb, "anchor": anchor, "T_t": Tt, "T_d": Td, "draft_tokens": x,
           "w1": torch.from_numpy(w1), "w2": torch.from_numpy(w2), "w1_f32": w1, "w2_f32": w2, "lengths": None}
    out, nacc = _run(cuda_lib, _torch_inputs(inp, lse), 5, 0)
    out, nacc = out.cpu().numpy(), nacc.cpu().numpy()

    def law(row):
        z = row.astype(np.float64) / 0.8
        p = np.exp(z - z.max())
        return p / p.sum()

    for sel, row in ((np.ones(B, bool), 0), (nacc >= 1, 1)):
        counts = np.bincount(out[sel, row], minlength=V)
        assert stats.chisquare(counts, sel.sum() * law(t[row]))[1] > 1e-4
    assert 0.05 < (nacc >= 1).mean() < 0.95
    rows = np.arange(0, B, 20)
    ref = _oracle(inp, 5, 0, rows)
    near = _compare(out, nacc, x, ref, V, GAP, rows)
    assert near <= len(rows) // 20


def test_bonus_only_and_all_greedy(cuda_lib):
    """lengths 0: the token is a draw from target row 0 (no draft row used); greedy drafts
    everywhere: no bias row is needed at all."""
    cfg = _small_cfg("bf16", 3001, 7, temps=(0.0,))
    inp = verify_logits_inputs(cfg)
    lse = oracle.draft_lse(inp["base_logits"], inp["anchor"], inp["w1_f32"], inp["w2_f32"], inp["T_d"],
                           inp["draft_tokens"])
    for lengths in (np.zeros(cfg.B, np.int32), None):
        inp["lengths"] = lengths
        out, nacc = _run(cuda_lib, _torch_inputs(inp, lse), 2, 9)
        ref = _oracle(inp, 2, 9)
        near = _compare(out.cpu().numpy(), nacc.cpu().numpy(), inp["draft_tokens"], ref, cfg.V, GAP)
        assert near <= 2
        if lengths is not None:
            assert np.all(nacc.cpu().numpy() == 0)


@pytest.mark.parametrize("B,gamma,V", [(12, 4, 1500), (64, 4, 70001)])
def test_invalid_requests_set_status(cuda_lib, B, gamma, V):
    """Out-of-range token, anchor or length, a non-positive target temperature, a negative draft
    temperature and a NaN draft lse each void their request (num_accepted 0, tokens -1) and set
    the status; the other requests still match the oracle.  The two sizes take the two row
    schedules (every drafted row in one round; one row per round)."""
    cfg = _small_cfg("bf16", V, 8, temps=(1.0,), B=B, gamma=gamma)
    inp = verify_logits_inputs(cfg)
    inp["lengths"] = np.full(cfg.B, cfg.gamma, np.int32)
    lse = oracle.draft_lse(inp["base_logits"], inp["anchor"], inp["w1_f32"], inp["w2_f32"], inp["T_d"],
                           inp["draft_tokens"]).astype(np.float32)
    good = np.ones(cfg.B, bool)
    inp["draft_tokens"][0, 0] = cfg.V + 5
    inp["anchor"][1] = -2
    inp["lengths"][2] = cfg.gamma + 1
    inp["T_t"][3] = 0.0
    inp["T_d"][4] = -1.0
    lse[5, 0] = np.nan
    good[:6] = False
    ws = cuda_lib.Workspace(cuda_lib.OP_VERIFY_LOGITS, cfg.B, cfg.gamma, cfg.V, cfg.r)
    out, nacc = _run(cuda_lib, _torch_inputs(inp, lse), 4, 0, workspace=ws)
    st, bits = cuda_lib.dspark_read_status(ws)
    out, nacc = out.cpu().numpy(), nacc.cpu().numpy()
    assert bits & cuda_lib.STATUS_INPUT_RANGE and bits & cuda_lib.STATUS_NUMERIC
    assert np.all(out[~good] == -1) and np.all(nacc[~good] == 0)
    rows = np.flatnonzero(good)
    ref = _oracle(inp, 4, 0, rows)
    assert _compare(out, nacc, inp["draft_tokens"], ref, cfg.V, GAP, rows) <= 1


def test_pipeline_from_the_sampler(cuda_lib):
    """The sampler's own tokens and lse feed verification (the path used in serving): the
    outputs are well formed and the status is clean."""
    import torch
    cfg = _small_cfg("bf16", 151936, 12, temps=(0.8,), r=256, B=16, gamma=8)
    inp = verify_logits_inputs(cfg)
    d = _torch_inputs(inp, np.zeros((cfg.B, cfg.gamma), np.float32))
    lse = torch.empty(cfg.B, cfg.gamma, dtype=torch.float32, device="cuda")
    x = cuda_lib.dspark_markov_sample(d["base_logits"], d["anchor"], d["w1"], d["w2"], d["T_d"], 7, 1, lse=lse)
    d["draft_tokens"], d["lse"] = x, lse
    ws = cuda_lib.Workspace(cuda_lib.OP_VERIFY_LOGITS, cfg.B, cfg.gamma, cfg.V, cfg.r)
    out, nacc = _run(cuda_lib, d, 3, 1, workspace=ws)
    st, bits = cuda_lib.dspark_read_status(ws)
    assert bits == 0
    out, nacc, x = out.cpu().numpy(), nacc.cpu().numpy(), x.cpu().numpy()
    lengths = inp["lengths"]
    for b in range(cfg.B):
        n = nacc[b]
        assert 0 <= n <= lengths[b] and np.all(out[b, :n] == x[b, :n])
        assert 0 <= out[b, n] < cfg.V and np.all(out[b, n + 1:] == -1)
