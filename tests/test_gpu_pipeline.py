"""GPU end-to-end draft step at the Qwen3-8B-shaped workload: base logits on the tensor
cores, then Markov sampling of the GPU's own logits, against the oracle's fp64 logits
and its own sampler run on the GPU's prefix (tokens equal except at near-ties of the perturbed
values, counted and bounded)."""
import numpy as np
import pytest

import oracle
from tests._helpers import check_markov_parity, to_dev
from workloads import DRAFT_CONFIGS, draft_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_draft_step_qwen3_8b_single(cuda_lib, T):
    import torch
    ds = cuda_lib
    cfg = DRAFT_CONFIGS["qwen3_8b_single"]
    inp = draft_inputs(cfg)
    Ts = np.full(cfg.B, T, np.float32)
    L = ds.dspark_draft_logits(to_dev(inp["hidden"]), to_dev(inp["lm_head"]))
    tok = ds.dspark_markov_sample(L.view(cfg.B, cfg.N, cfg.V), to_dev(inp["anchor"]), to_dev(inp["w1"]),
                                  to_dev(inp["w2"]), to_dev(Ts), 0, 0)
    torch.cuda.synchronize()
    L_ref = oracle.draft_logits(inp["hidden_f32"], inp["lm_head_f32"]).reshape(cfg.B, cfg.N, cfg.V)
    check_markov_parity(tok.cpu().numpy(), L_ref, inp["anchor"], inp["w1_f32"], inp["w2_f32"], Ts, 0, 0,
                        label=f"pipeline qwen3_8b_single T={T}", kind="markov (GPU logits)")
