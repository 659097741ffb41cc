"""Cases run through both builds of the library by tests/test_gpu_checked.py: the default build
(this process) and the DSPARK_CHECKED build (a child process that loads it through
DSPARK_LIBRARY).  Each case returns its outputs and the raw status bits of its workspace.

Clean cases must leave no status bit in either build.  Planted cases put one caller index out of
range (an anchor, a draft token, a draft-to-target table entry); both builds substitute the same
safe value and flag INPUT_RANGE, and only the checked build adds INDEX.  No case reads memory at
an out-of-range index in either build: every planted index is one the kernels check
unconditionally.
"""
import json
import sys

import numpy as np


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _markov_inputs(B, N, V, r, seed):
    rng = np.random.default_rng(seed)
    L = (rng.standard_normal((B, N, V)) * 2).astype(np.float32)
    w1 = rng.standard_normal((V, r)).astype(np.float32)
    w2 = (rng.standard_normal((V, r)) / np.sqrt(r)).astype(np.float32)
    anchor = rng.integers(0, V, B).astype(np.int32)
    T = np.full(B, 1.0, np.float32)
    return L, w1, w2, anchor, T


def _bf16(a):
    import torch
    return torch.from_numpy(a).to(torch.bfloat16).cuda()


def run_cases(ds):
    import torch
    out = {}

    def status(ws):
        return int(ds.dspark_read_status(ws)[1])

    # Markov sampler, CUDA-core path (fp32 head): clean, then anchor 1 out of range
    B, N, V, r = 3, 4, 5000, 24
    L, w1, w2, anchor, T = _markov_inputs(B, N, V, r, 1)
    for name, anc in (("markov_clean", anchor), ("markov_anchor", np.array([anchor[0], V + 5, anchor[2]], np.int32))):
        ws = ds.Workspace(ds.OP_MARKOV_SAMPLE, B, N, V, r)
        tok = ds.dspark_markov_sample(_dev(L), _dev(anc), _dev(w1), _dev(w2), _dev(T), 7, 0, workspace=ws)
        out[name] = {"bits": status(ws), "tokens": tok.cpu().numpy().tolist()}

    # Markov sampler, tensor-core path (bf16 head, r = 256, a batch): clean, then anchor 5 negative
    B, N, V, r = 20, 3, 8192, 256
    L, w1, w2, anchor, T = _markov_inputs(B, N, V, r, 2)
    tw1, tw2 = _bf16(w1), _bf16(w2)
    for name, anc in (("markov_tc_clean", anchor), ("markov_tc_anchor", np.where(np.arange(B) == 5, -2, anchor))):
        ws = ds.Workspace(ds.OP_MARKOV_SAMPLE, B, N, V, r)
        tok = ds.dspark_markov_sample(_dev(L), _dev(anc.astype(np.int32)), tw1, tw2, _dev(T), 3, 1, workspace=ws)
        out[name] = {"bits": status(ws), "tokens": tok.cpu().numpy().tolist()}

    # reduced draft vocabulary: one table entry maps outside the target vocabulary
    B, N, Vd, r, Vt = 2, 3, 3000, 16, 50000
    L, w1, w2, anchor, T = _markov_inputs(B, N, Vd, r, 3)
    d2t = np.sort(np.random.default_rng(3).choice(Vt, Vd, replace=False)).astype(np.int32)
    ws = ds.Workspace(ds.OP_MARKOV_SAMPLE, B, N, Vd, r)
    tok = ds.dspark_markov_sample_reduced(_dev(L), _dev(anchor), _dev(w1), _dev(w2), _dev(T), 5, 0, _dev(d2t),
                                          ds.D2T_INDEX, Vt, workspace=ws)
    clean = tok.cpu().numpy()
    out["reduced_clean"] = {"bits": status(ws), "tokens": clean.tolist()}
    bad = d2t.copy()
    drafted = np.searchsorted(d2t, clean[0, 1])           # the draft id behind request 0, step 1
    bad[drafted] = Vt + 100
    tok = ds.dspark_markov_sample_reduced(_dev(L), _dev(anchor), _dev(w1), _dev(w2), _dev(T), 5, 0, _dev(bad),
                                          ds.D2T_INDEX, Vt, workspace=ws)
    out["reduced_table"] = {"bits": status(ws), "tokens": tok.cpu().numpy().tolist()}

    # verification: clean, then one draft token out of range
    B, g, V = 4, 4, 1000
    rng = np.random.default_rng(4)
    pt = rng.dirichlet(np.ones(V), size=(B, g + 1)).astype(np.float32)
    pd = rng.dirichlet(np.ones(V), size=(B, g)).astype(np.float32)
    toks = rng.integers(0, V, (B, g)).astype(np.int32)
    for name, tk in (("verify_clean", toks), ("verify_token", np.where((np.arange(B)[:, None] == 2) &
                                                                        (np.arange(g)[None] == 1), -3, toks))):
        ws = ds.Workspace(ds.OP_VERIFY, B, g, V)
        o, nacc = ds.dspark_verify(_dev(pt), _dev(pd), _dev(tk.astype(np.int32)), None, 11, 0, workspace=ws)
        out[name] = {"bits": status(ws), "tokens": o.cpu().numpy().tolist(), "accepted": nacc.cpu().numpy().tolist()}

    # confidence head: clean, then one draft token out of range
    B, N, H, V, r = 2, 5, 64, 700, 16
    rng = np.random.default_rng(5)
    hid = rng.standard_normal((B * N, H)).astype(np.float32)
    w1 = rng.standard_normal((V, r)).astype(np.float32)
    anchor = rng.integers(0, V, B).astype(np.int32)
    toks = rng.integers(0, V, (B, N)).astype(np.int32)
    w_h = (rng.standard_normal(H) / 8).astype(np.float32)
    w_e = (rng.standard_normal(r) / 4).astype(np.float32)
    tau = np.full(N, 1.1, np.float32)
    for name, tk in (("confidence_clean", toks), ("confidence_token", np.where(np.arange(N)[None] == 2, V, toks))):
        ws = ds.Workspace(ds.OP_CONFIDENCE, B, N, V, r)
        c = ds.dspark_confidence(_dev(hid), _dev(w1), _dev(anchor), _dev(tk.astype(np.int32)), _dev(w_h), _dev(w_e),
                                 0.25, _dev(tau), workspace=ws)
        out[name] = {"bits": status(ws), "conf": c.cpu().numpy().tolist()}

    # admission pools through every scheduler kernel (warp, one block, cluster, workspace keys)
    for B, N in ((2, 16), (64, 16), (1024, 16), (1100, 16)):
        rng = np.random.default_rng(B)
        c = rng.beta(4, 1.5, size=(B, N)).astype(np.float32)
        sps = (100.0 * (1 + 0.05 * np.cos(np.arange(B * N)))).astype(np.float64)
        ws = ds.Workspace(ds.OP_SCHEDULE, B, N)
        surv, K, lengths, sel = ds.dspark_schedule(_dev(c), _dev(sps), -1, workspace=ws)
        out[f"schedule_{B}x{N}"] = {"bits": status(ws), "K": int(K.item()), "lengths": lengths.cpu().numpy().tolist(),
                                    "selected": sel.cpu().numpy().tolist()}
    torch.cuda.synchronize()
    return out


if __name__ == "__main__":
    sys.path.insert(0, sys.argv[2])
    import draft_sampling_verification_tcgen05_gb300 as ds_checked
    res = run_cases(ds_checked)
    res["_library"] = ds_checked.LIB_PATH
    with open(sys.argv[1], "w") as f:
        json.dump(res, f)
