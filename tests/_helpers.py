"""Helpers shared by the GPU parity tests (comparison rules, device transfer)."""
import numpy as np

NEAR_TIE = 5e-2           # top-2 perturbed-logit gap below which a token may differ
LOGIT_TOL = 2e-2          # max abs error of base logits (bf16 inputs, fp32 accumulation)


def to_dev(a, dev="cuda"):
    import torch
    if isinstance(a, np.ndarray):
        a = torch.from_numpy(np.ascontiguousarray(a))
    return a.to(dev)


def compare_markov_tokens(gpu_tokens, ref_tokens, ref_gap, near_tie=NEAR_TIE):
    """Free-running comparison of two token sequences per request.

    Tokens must agree position by position.  The first disagreement of a request
    is allowed only where the oracle's top-2 gap of perturbed values is below
    `near_tie` (an fp32-vs-fp64 rounding can flip such a tie); later positions of
    that request are then conditioned on different prefixes and are not compared.
    Returns (compared positions, near-tie divergences); raises on a real mismatch.
    """
    g = np.asarray(gpu_tokens)
    r = np.asarray(ref_tokens)
    B, N = r.shape
    compared = ties = 0
    for b in range(B):
        for i in range(N):
            compared += 1
            if g[b, i] != r[b, i]:
                assert ref_gap[b, i] < near_tie, (
                    f"token mismatch at request {b} step {i}: gpu {g[b, i]} oracle {r[b, i]} "
                    f"(oracle top-2 gap {ref_gap[b, i]:.3g} >= {near_tie})")
                ties += 1
                break
    return compared, ties
