"""Verification with the draft's own Gumbel noise (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "DSpark implementation and evaluation" §5 (probabilistic draft
sampling): the draft turns its logits into tokens with the Gumbel-max trick,
and the target verifies with the same Gumbel seed, which keeps the output
distribution unchanged.

Reading (the page gives no more than that sentence): the target draws its own
token at each drafted position with the Gumbel-max trick on the very noise the
draft used at that position -- y_k = argmax_v (t[b, k, v] / T_b + g(b, k, v)),
g the draft noise of draft step k for request b (``philox.draft_gumbel`` with
the draft sampler's seed and offset).  Draft token x_k is accepted while
x_k = y_k; at the first position k* where they differ, y_{k*} is emitted
instead; when every tested token is accepted, y_{L_b} is the bonus token.  The
emitted tokens are then exactly the target's own Gumbel-max samples, so their
law is the target's (the noise of position k is independent of everything that
decided the prefix); the draft only decides how many of them come for free.
With T_b = 0 the target token is the plain argmax (greedy verification).

Other readings, as in the other verifications: row k of the target input
[B, gamma+1, V] scores position k; ties go to the lowest id; NaN never wins; a
length L_b <= gamma truncates the block; a token outside [0, V) or a length
outside [0, gamma] makes the request invalid (nothing accepted, -1 fill).
"""
from __future__ import annotations

import numpy as np

from .philox import draft_gumbel


def _scored_argmax(r: np.ndarray):
    """Row-wise argmax (lowest index on ties, NaN never chosen, 0 for an all-NaN row) and the
    top-2 gap (inf with fewer than two non-NaN entries) of r [n, V]."""
    s = np.where(np.isnan(r), -np.inf, r)
    tok = np.argmax(s, axis=1)
    rows = np.arange(s.shape[0])
    top = s[rows, tok]
    s2 = s.copy()
    s2[rows, tok] = -np.inf
    second = s2.max(axis=1) if s.shape[1] > 1 else np.full(s.shape[0], -np.inf)
    gap = np.where(np.isfinite(second) & np.isfinite(top), top - second, np.inf)
    return np.where(np.isfinite(top), tok, 0), gap


def target_gumbel_tokens(target_logits: np.ndarray, temperature: np.ndarray, seed: int, offset: int,
                         req_ids=None, noise=None):
    """The target's token at every position: y[b, k] = argmax_v (t[b, k, v] / T_b + g(b, k, v)),
    g the draft noise of draft step k for request req_ids[b] (plain argmax where T_b = 0).
    noise(k, request ids) -> [n, V] replaces the Philox draft noise (hand-worked tests).
    Returns (y [B, gamma+1] int64, gap [B, gamma+1] float64 top-2 gaps of the scored rows)."""
    t = np.asarray(target_logits, dtype=np.float64)
    T = np.asarray(temperature, dtype=np.float64)
    B, g1, V = t.shape
    req = np.arange(B) if req_ids is None else np.asarray(req_ids)
    hot = T > 0
    y = np.zeros((B, g1), dtype=np.int64)
    gap = np.full((B, g1), np.inf)
    for k in range(g1):
        r = t[:, k, :].copy()
        if hot.any():
            g = draft_gumbel(seed, offset, req[hot], k, V) if noise is None else noise(k, req[hot])
            r[hot] = r[hot] / T[hot, None] + g
        y[:, k], gap[:, k] = _scored_argmax(r)
    return y, gap


def verify_gumbel(target_logits: np.ndarray, temperature: np.ndarray, draft_tokens: np.ndarray,
                  seed: int, offset: int, lengths=None, return_gaps: bool = False, req_ids=None, noise=None):
    """Returns (out_tokens [B, gamma+1] int64, num_accepted [B] int64), and with return_gaps the
    smallest top-2 gap over the rows each request's result depends on (rows 0..k*; inf for an
    invalid request).  req_ids: the request index of each row in the draft batch (the noise
    counter), default 0..B-1."""
    x = np.asarray(draft_tokens, dtype=np.int64)
    B, g1, V = np.asarray(target_logits).shape
    gamma = g1 - 1
    y, gap = target_gumbel_tokens(target_logits, temperature, seed, offset, req_ids, noise)
    out = np.full((B, gamma + 1), -1, dtype=np.int64)
    nacc = np.zeros(B, dtype=np.int64)
    gaps = np.full(B, np.inf)
    for b in range(B):
        L = gamma if lengths is None else int(lengths[b])
        if not 0 <= L <= gamma or np.any((x[b, :L] < 0) | (x[b, :L] >= V)):
            continue
        k = 0
        while k < L and x[b, k] == y[b, k]:              # accepted while the target draws the same token
            k += 1
        out[b, :k] = x[b, :k]
        out[b, k] = y[b, k]                               # the target's own token at the first mismatch
        nacc[b] = k
        gaps[b] = gap[b, :k + 1].min()
    return (out, nacc, gaps) if return_gaps else (out, nacc)
