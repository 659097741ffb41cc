"""Greedy (temperature-0) verification of a drafted block (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "xserv/docs/25-speculative-methods-comparison.md" §2 (small-model
speculative decoding): the target scores all drafted positions in one forward
pass; the longest prefix of draft tokens that each equal the target's argmax
at their position is accepted, and the target's argmax at the first
position that fails (the position after the block when none fails) is
appended as the correction.  The output is then exactly the target's own
greedy continuation.

Readings:
  * row k of the target input [B, gamma+1, V] scores position k (the same
    convention as the stochastic verification: row k pairs with draft token
    x_k, row gamma is the position after the block); the rows may be logits
    or probabilities -- only their argmax matters;
  * argmax ties go to the lowest token id; NaN entries never win (a row with
    no non-NaN entry gives token 0);
  * a per-request length L_b <= gamma truncates the block: only x_0..x_{L_b-1}
    are tested and the correction of a fully accepted block comes from row L_b;
  * a token outside [0, V) or a length outside [0, gamma] makes the request
    invalid: no token accepted, every output -1 (the GPU also raises a flag).
"""
from __future__ import annotations

import numpy as np


def row_argmax(row: np.ndarray) -> int:
    """Index of the largest entry, lowest index on ties, NaN never chosen (0 if all NaN)."""
    r = np.asarray(row, dtype=np.float64)
    r = np.where(np.isnan(r), -np.inf, r)
    if np.all(r == -np.inf):
        return 0
    return int(np.argmax(r))


def verify_greedy(target: np.ndarray, draft_tokens: np.ndarray, lengths=None):
    """Returns (out_tokens [B, gamma+1] int64, num_accepted [B] int64)."""
    target = np.asarray(target)
    x = np.asarray(draft_tokens, dtype=np.int64)
    B, g1, V = target.shape
    gamma = g1 - 1
    out = np.full((B, gamma + 1), -1, dtype=np.int64)
    nacc = np.zeros(B, dtype=np.int64)
    for b in range(B):
        L = gamma if lengths is None else int(lengths[b])
        if not 0 <= L <= gamma or np.any((x[b, :L] < 0) | (x[b, :L] >= V)):
            continue                                   # invalid request: nothing accepted, -1 fill
        k = 0
        while k < L and x[b, k] == row_argmax(target[b, k]):
            k += 1
        out[b, :k] = x[b, :k]
        out[b, k] = row_argmax(target[b, k])
        nacc[b] = k
    return out, nacc
