"""GPU parity: Markov sampling on a reduced draft vocabulary, tokens returned as target ids.

Compared with the oracle at every position on the GPU's own prefix (teacher forcing; same
near-tie rule and bound as the plain sampler), on the CUDA-core path
(one request, EAGLE-3-sized 32000-entry draft vocabulary in a 151936-entry target vocabulary)
and on the tensor-core path; both table conventions; identity tables reproduce the plain
sampler exactly; unmappable ids come back as -1 with a flag."""
import numpy as np
import pytest

import oracle
from oracle.reduced_vocab import MODE_INDEX, MODE_OFFSET
from tests._helpers import check_tie_share, compare_teacher_forced, record_parity, to_dev
from workloads import DraftConfig, markov_logits, normal_rows, to_bf16_values

pytestmark = pytest.mark.gpu
V_TARGET = 151936


def _case(B, N, Vd, r, seed):
    cfg = DraftConfig("red", B=B, N=N, H=8, V=Vd, r=r, dtype="bf16", temperatures=(1.0,), data_seed=seed)
    L = markov_logits(cfg, scale=2.0)
    tw1, w1 = to_bf16_values(normal_rows(Vd, r, 1.0, seed, "w1"))
    tw2, w2 = to_bf16_values(normal_rows(Vd, r, 1.0 / np.sqrt(r), seed, "w2"))
    rng = np.random.default_rng(seed)
    anchor = rng.integers(0, Vd, B).astype(np.int32)
    table = np.sort(rng.choice(V_TARGET, Vd, replace=False)).astype(np.int32)
    return L, tw1, w1, tw2, w2, anchor, table


@pytest.mark.parametrize("B,N,Vd,r,T", [(1, 8, 32000, 64, 1.0), (3, 5, 32000, 64, 0.0), (32, 4, 32000, 256, 0.8)])
@pytest.mark.parametrize("mode", [MODE_INDEX, MODE_OFFSET])
def test_matches_oracle(cuda_lib, B, N, Vd, r, T, mode):
    L, tw1, w1, tw2, w2, anchor, table = _case(B, N, Vd, r, 40 + B)
    d2t = table if mode == MODE_INDEX else (table - np.arange(Vd)).astype(np.int32)
    Ts = np.full(B, T, np.float32)
    tok = cuda_lib.dspark_markov_sample_reduced(to_dev(L), to_dev(anchor), to_dev(tw1), to_dev(tw2), to_dev(Ts),
                                                6, 2, to_dev(d2t), mode, V_TARGET).cpu().numpy()
    assert np.all(np.isin(tok, table))
    draft_ids = np.searchsorted(table, tok)             # the table is strictly increasing
    ref_t, ref_d, gap, _ = oracle.markov_sample_reduced(L, anchor, w1, w2, Ts, 6, 2, d2t, mode, V_TARGET,
                                                        forced_draft_tokens=draft_ids)
    n, ties = compare_teacher_forced(draft_ids, ref_d, gap)
    check_tie_share(n, ties, f"reduced B={B} mode={mode}")
    record_parity("markov reduced vocabulary", f"B={B} N={N} mode={mode}", n, ties)
    np.testing.assert_array_equal(tok[draft_ids == ref_d], ref_t[draft_ids == ref_d])


def test_identity_table_reproduces_the_plain_sampler(cuda_lib):
    L, tw1, w1, tw2, w2, anchor, _ = _case(16, 3, 4096, 64, 7)
    Ts = np.full(16, 0.9, np.float32)
    args = (to_dev(L), to_dev(anchor), to_dev(tw1), to_dev(tw2), to_dev(Ts), 1, 0)
    plain = cuda_lib.dspark_markov_sample(*args).cpu().numpy()
    ident = cuda_lib.dspark_markov_sample_reduced(*args, to_dev(np.arange(4096, dtype=np.int32)), MODE_INDEX,
                                                  4096).cpu().numpy()
    zero = cuda_lib.dspark_markov_sample_reduced(*args, to_dev(np.zeros(4096, np.int32)), MODE_OFFSET,
                                                 4096).cpu().numpy()
    np.testing.assert_array_equal(ident, plain)
    np.testing.assert_array_equal(zero, plain)


def test_unmappable_ids_are_minus_one_and_flagged(cuda_lib):
    L, tw1, w1, tw2, w2, anchor, _ = _case(2, 3, 1000, 16, 8)
    Ts = np.ones(2, np.float32)
    ws = cuda_lib.Workspace(cuda_lib.OP_MARKOV_SAMPLE, 2, 3, 1000, 16)
    tok = cuda_lib.dspark_markov_sample_reduced(to_dev(L), to_dev(anchor), to_dev(tw1), to_dev(tw2), to_dev(Ts),
                                                0, 0, to_dev(np.full(1000, 5000, np.int32)), MODE_INDEX, 4000,
                                                workspace=ws).cpu().numpy()
    st, bits = cuda_lib.dspark_read_status(ws)
    assert np.all(tok == -1) and bits & cuda_lib.STATUS_INPUT_RANGE
