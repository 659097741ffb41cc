"""All four calls can be captured into one CUDA graph (fixed buffers, no allocation or
host synchronisation inside the calls) and replayed with identical results."""
import numpy as np
import pytest

from tests._helpers import to_dev
from workloads import (DRAFT_CONFIGS, VERIFY_CONFIGS, SCHEDULE_CONFIGS, draft_inputs, verify_inputs,
                       schedule_inputs)

pytestmark = pytest.mark.gpu


def test_capture_and_replay_whole_step(cuda_lib):
    import torch
    ds = cuda_lib
    cfg = DRAFT_CONFIGS["tiny"]
    inp = draft_inputs(cfg)
    X, W = to_dev(inp["hidden"]), to_dev(inp["lm_head"])
    anchor, w1, w2 = to_dev(inp["anchor"]), to_dev(inp["w1"]), to_dev(inp["w2"])
    T = torch.ones(cfg.B, device="cuda")
    vin = verify_inputs(VERIFY_CONFIGS["tiny"])
    p_t, p_d = to_dev(vin["p_t"]), to_dev(vin["p_d"])
    sin = schedule_inputs(SCHEDULE_CONFIGS["tiny"])
    c, sps = to_dev(sin["cond_accept"]), to_dev(sin["sps"])

    L = torch.empty(cfg.B * cfg.N, cfg.V, device="cuda")
    tok = torch.empty(cfg.B, cfg.N, dtype=torch.int32, device="cuda")
    out = torch.empty(1, 9, dtype=torch.int32, device="cuda")
    nacc = torch.empty(1, dtype=torch.int32, device="cuda")
    surv = torch.empty(1, 8, device="cuda")
    K = torch.empty(1, dtype=torch.int32, device="cuda")
    lens = torch.empty(1, dtype=torch.int32, device="cuda")
    sel = torch.empty(8, dtype=torch.int32, device="cuda")
    ws_g = ds.Workspace(ds.OP_DRAFT_LOGITS)
    ws_m = ds.Workspace(ds.OP_MARKOV_SAMPLE, cfg.B, cfg.N, cfg.V, cfg.r)
    ws_v = ds.Workspace(ds.OP_VERIFY, 1, 8, cfg.V)
    ws_s = ds.Workspace(ds.OP_SCHEDULE, 1, 8)

    def step():
        ds.dspark_draft_logits(X, W, logits=L, workspace=ws_g)
        ds.dspark_markov_sample(L.view(cfg.B, cfg.N, cfg.V), anchor, w1, w2, T, 0, 0, draft_tokens=tok,
                                workspace=ws_m)
        ds.dspark_verify(p_t, p_d, tok, None, 2, 0, out_tokens=out, num_accepted=nacc, workspace=ws_v)
        ds.dspark_schedule(c, sps, -1, survival=surv, K_out=K, lengths=lens, selected=sel, workspace=ws_s)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (L, tok, out, nacc, surv, K, lens, sel)]
    for t in (L, tok, out, nacc, surv, K, lens, sel):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, (L, tok, out, nacc, surv, K, lens, sel)):
        assert torch.equal(a, b)
