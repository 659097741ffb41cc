"""Lossless verification from logits, with the draft distribution recomputed (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources:
  * "Speculative decoding: from zero to DSpark" (bittide.aicompass.dev) §2 --
    the rejection rule: accept x_k with probability min(1, p_t(x_k)/p_d(x_k)),
    at the first rejection draw from norm(max(0, p_t - p_d)), after a fully
    accepted block draw a bonus token from p_t of the next position;
  * "DSpark implementation and evaluation" §2.2 / §5 -- the draft distribution
    of position k is the one the Gumbel-max sampler draws from,
    softmax((base_logits[:, k] + markov_w2 . markov_w1[prev]) / T), and the
    probabilistic mode verifies against it without keeping draft
    probabilities around.

Readings:
  * target distribution of row k: softmax(target_logits[b, k] / T_t[b]), T_t > 0;
    draft distribution of position k: softmax(z) with z as above, prev = anchor
    for k = 0 and x_{k-1} after; a greedy draft (T_d = 0) has the point mass at
    its token as its distribution;
  * the acceptance test is the one of ``verify``: fl32(u_k * p_d(x_k)) < p_t(x_k)
    on the float32 roundings of the two probabilities, u_k the stream-1 uniform;
  * the correction / bonus token is drawn by Gumbel-max: argmax_v of
    log w_v + g_v with w = max(0, p_t - p_d) (rejection) or p_t (bonus) and g_v
    the standard Gumbel variate of stream 4, word v & 3 of counter
    (v >> 2, b, (4 << 16) | position, offset); entries with w_v = 0 never win;
    a residual with no positive entry falls back to w = p_t.  This has the law
    of the rule (Gumbel-max draws v with probability w_v / sum w).  The integer
    inverse CDF of ``verify`` is not used here: recomputed probabilities carry
    the rounding of their normalisers, which moves every CDF boundary by about
    1e-7 of the total mass, as much as one entry's width at V ~ 1.5e5, while
    the Gumbel-max decision depends on the gap between the two largest
    perturbed values, of order one;
  * everything is float64 here; the device computes in float32, so the two may
    part only where a decision sits within rounding of its boundary: every
    request reports the smallest relative margin of its acceptance tests and
    the top-2 gap of its draw.
"""
from __future__ import annotations

import numpy as np

from .draft import markov_bias
from .philox import philox_words, gumbel_from_word, STREAM_RESIDUAL
from .verify import verify_draws


def _softmax(z: np.ndarray) -> np.ndarray:
    m = z.max(axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=-1, keepdims=True)


def _logsumexp(z: np.ndarray) -> np.ndarray:
    m = z.max(axis=-1)
    return m + np.log(np.exp(z - m[..., None]).sum(axis=-1))


def _prev_tokens(anchor, draft_tokens):
    x = np.asarray(draft_tokens, dtype=np.int64)
    return np.concatenate([np.asarray(anchor, dtype=np.int64).reshape(-1, 1), x[:, :-1]], axis=1)


def draft_distributions(base_logits, anchor, w1, w2, T_d, draft_tokens):
    """p_d [B, gamma, V] float64: the sampler's distribution at each drafted position."""
    L = np.asarray(base_logits, dtype=np.float64)
    B, gamma, V = L.shape
    x = np.asarray(draft_tokens, dtype=np.int64)
    prev = _prev_tokens(anchor, x)
    T = np.asarray(T_d, dtype=np.float64).reshape(B)
    p = np.zeros_like(L)
    for k in range(gamma):
        hot = T == 0
        if (~hot).any():
            rows = np.flatnonzero(~hot)
            z = (L[rows, k] + markov_bias(prev[rows, k], w1, w2)) / T[rows, None]
            p[rows, k] = _softmax(z)
        p[np.flatnonzero(hot), k, x[hot, k]] = 1.0
    return p


def draft_lse(base_logits, anchor, w1, w2, T_d, draft_tokens):
    """[B, gamma] float64: log-sum-exp of z at each drafted position -- what the sampler
    reports as its lse output when it drew these tokens (T_d = 0: of base + bias)."""
    L = np.asarray(base_logits, dtype=np.float64)
    B, gamma, V = L.shape
    prev = _prev_tokens(anchor, draft_tokens)
    T = np.asarray(T_d, dtype=np.float64).reshape(B)
    scale = np.where(T > 0, T, 1.0)
    out = np.empty((B, gamma))
    for k in range(gamma):
        out[:, k] = _logsumexp((L[:, k] + markov_bias(prev[:, k], w1, w2)) / scale[:, None])
    return out


def residual_gumbel(seed: int, offset: int, b, k: int, V: int) -> np.ndarray:
    """Gumbel variates g_v (v < V) of the resample draw of request b at position k."""
    v = np.arange(V, dtype=np.uint64)
    words = philox_words(seed, offset, v >> np.uint64(2), np.uint64(b), STREAM_RESIDUAL, np.uint64(k))
    w = np.choose((v & np.uint64(3)).astype(np.int64), words)
    return gumbel_from_word(w)


def verify_from_logits(target_logits, T_t, base_logits, anchor, w1, w2, T_d, draft_tokens, lengths,
                       seed: int, offset: int, req_ids=None):
    """Verification of drafted blocks from the target's logits and the draft's base logits.

    target_logits [B, gamma+1, V], T_t [B] (> 0), base_logits [B, gamma, V] (the
    drafted positions' base logits), anchor [B], w1 / w2 [V, r], T_d [B] (>= 0),
    draft_tokens [B, gamma], lengths [B] or None (all gamma).  req_ids: request
    index used in the random-number counters (default 0..B-1).

    Returns (out_tokens [B, gamma+1] int64, num_accepted [B] int64,
             accept_margin [B], draw_gap [B]) where accept_margin is the smallest
    |u p_d(x) - p_t(x)| / p_t(x) over the tests made and draw_gap the difference
    of the two largest perturbed values of the draw (inf if only one entry competes).
    """
    t = np.asarray(target_logits, dtype=np.float64)
    B, g1, V = t.shape
    gamma = g1 - 1
    x = np.asarray(draft_tokens, dtype=np.int64)
    req = np.arange(B) if req_ids is None else np.asarray(req_ids)
    Lb = np.full(B, gamma, dtype=np.int64) if lengths is None else np.asarray(lengths, np.int64)
    Tt = np.asarray(T_t, dtype=np.float64).reshape(B)
    p_t = _softmax(t / Tt[:, None, None])
    p_d = draft_distributions(base_logits, anchor, w1, w2, T_d, x)
    u, _ = verify_draws(B, gamma, seed, offset, req)

    out = np.full((B, g1), -1, dtype=np.int64)
    n_acc = np.zeros(B, dtype=np.int64)
    acc_margin = np.full(B, np.inf)
    draw_gap = np.full(B, np.inf)
    for b in range(B):
        kstar = int(Lb[b])
        for k in range(int(Lb[b])):
            pt = np.float32(p_t[b, k, x[b, k]])
            pd = np.float32(p_d[b, k, x[b, k]])
            prod = np.float32(u[b, k] * pd)                       # u is a float32 value
            acc_margin[b] = min(acc_margin[b], abs(float(u[b, k]) * p_d[b, k, x[b, k]] - p_t[b, k, x[b, k]])
                                / max(p_t[b, k, x[b, k]], 1e-300))
            if not prod < pt:
                kstar = k
                break
        if kstar < Lb[b]:
            w = np.maximum(0.0, p_t[b, kstar] - p_d[b, kstar])
            if not (w > 0).any():
                w = p_t[b, kstar]
        else:
            w = p_t[b, kstar]
        gv = residual_gumbel(seed, offset, req[b], kstar, V)
        with np.errstate(divide="ignore"):
            y = np.where(w > 0, np.log(w) + gv, -np.inf)
        order = np.argsort(-y, kind="stable")
        top = int(order[0])
        if V > 1 and np.isfinite(y[order[1]]):
            draw_gap[b] = float(y[order[0]] - y[order[1]])
        out[b, :kstar] = x[b, :kstar]
        out[b, kstar] = top
        n_acc[b] = kstar
    return out, n_acc, acc_margin, draw_gap
