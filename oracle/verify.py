"""Lossless speculative verification (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "Speculative decoding: from zero to DSpark" (bittide.aicompass.dev) §2:
the target checks the drafted block left to right; draft token x_k is accepted
with probability min(1, p_t(x_k) / p_d(x_k)); at the first rejection a
correction token is drawn from norm(max(0, p_t - p_d)); if every drafted token
is accepted, a bonus token is drawn from the target distribution of the
position after the block.  The per-position acceptance probability equals
1 - TV(p_t, p_d).

Readings (the pages give the rule, not its arithmetic):
  * inputs are float32 probabilities; "accept with probability
    min(1, p_t/p_d)" is decided as  fl32(u_k * p_d[x_k]) < p_t[x_k]  with u_k the
    stream-1 uniform of position k (this also covers p_d[x_k] = 0);
  * the residual max(0, p_t - p_d) is formed in float32 (one rounded
    subtraction), quantised to q_v = floor(w_v * 2**40) as an integer, and
    sampled by inverse CDF: with R the 64-bit stream-2 word pair and
    Q = sum q_v, t = floor(R * Q / 2**64) and the token is the smallest v whose
    inclusive prefix sum of q exceeds t.  Integer sums make the result
    independent of summation order;
  * if the residual has no mass (only float32 rounding can cause it), the
    row p_t itself is used; if that too has no mass, the token is argmax p_t
    and the numeric flag is raised;
  * a per-request length L_b <= gamma (from the scheduler) truncates the block:
    only x_0..x_{L_b-1} are tested and the bonus comes from position L_b.
"""
from __future__ import annotations

import numpy as np

from .philox import philox_words, uniform_from_word, STREAM_ACCEPT, STREAM_RESAMPLE

TWO40 = float(2 ** 40)


def _quantise(w: np.ndarray) -> np.ndarray:
    """q_v = floor(w_v * 2**40) for float32 w_v in [0, 1] (exact: scaling by a power of two)."""
    return np.floor(np.asarray(w, dtype=np.float64) * TWO40).astype(np.uint64)


def verify_draws(B: int, gamma: int, seed: int, offset: int, req_ids=None):
    """The method's random draws: u [B, gamma] (float32 values) and R [B, gamma+1] (Python ints).

    u[b, k] is the stream-1 uniform of position k; R[b, k] = (w0 << 32) | w1 of
    the stream-2 counter of position k (used at the first rejection k, or at
    the bonus position L_b).
    """
    req = np.arange(B) if req_ids is None else np.asarray(req_ids)
    k = np.arange(gamma + 1, dtype=np.uint64)[None, :]
    b = req.astype(np.uint64)[:, None]
    wa = philox_words(seed, offset, 0, b, STREAM_ACCEPT, k[:, :gamma])[0]
    u = uniform_from_word(wa).astype(np.float32)
    wr = philox_words(seed, offset, 0, b, STREAM_RESAMPLE, k)
    R = (wr[0].astype(object) << 32) | wr[1].astype(object)
    return u, R


def verify_given_draws(p_target, p_draft, draft_tokens, lengths, u, R):
    """The verification rule with the random draws supplied (see verify_draws).

    Returns (out_tokens [B, gamma+1] int64, num_accepted [B] int64,
             accept [B, gamma] int8 (1 accepted, 0 rejected, -1 not tested),
             numeric [B] bool).
    """
    p_t = np.asarray(p_target, dtype=np.float32)
    p_d = np.asarray(p_draft, dtype=np.float32)
    x = np.asarray(draft_tokens, dtype=np.int64)
    B, gamma, V = p_d.shape
    Lb = np.full(B, gamma, dtype=np.int64) if lengths is None else np.asarray(lengths, np.int64)
    rows = np.arange(B)

    # ratio test at every position, then the first rejection
    kk = np.arange(gamma)[None, :]
    pd_x = p_d[rows[:, None], kk, x]
    pt_x = p_t[rows[:, None], kk, x]
    ok = (np.asarray(u, np.float32) * pd_x).astype(np.float32) < pt_x
    tested = kk < Lb[:, None]
    rejected = tested & ~ok
    kstar = np.where(rejected.any(axis=1), rejected.argmax(axis=1), Lb)
    accept = np.where(tested & (kk <= kstar[:, None]), ok.astype(np.int8), np.int8(-1))

    # residual (rejection) or bonus row, in float32
    is_rej = kstar < Lb
    w = p_t[rows, kstar].copy()
    w[is_rej] = np.maximum(np.float32(0), p_t[rows[is_rej], kstar[is_rej]]
                           - p_d[rows[is_rej], kstar[is_rej]])
    q = _quantise(w)
    Q = q.sum(axis=1, dtype=np.uint64)
    redo = is_rej & (Q == 0)
    if redo.any():
        q[redo] = _quantise(p_t[rows[redo], kstar[redo]])
        Q = q.sum(axis=1, dtype=np.uint64)
    numeric = Q == 0

    # inverse CDF: t = floor(R * Q / 2**64) in exact integers, token = first v with prefix > t
    R_sel = np.asarray(R, dtype=object)[rows, kstar]
    t = np.asarray((R_sel * Q.astype(object)) >> 64, dtype=np.uint64)
    csum = np.cumsum(q, axis=1, dtype=np.uint64)
    y = np.argmax(csum > t[:, None], axis=1)
    if numeric.any():
        y[numeric] = np.argmax(p_t[rows[numeric], kstar[numeric]], axis=1)
    out = np.full((B, gamma + 1), -1, dtype=np.int64)
    out[:, :gamma] = np.where(kk < kstar[:, None], x, -1)     # the accepted prefix
    out[rows, kstar] = y                                        # then the correction / bonus
    return out, kstar, accept, numeric


def verify(p_target, p_draft, draft_tokens, lengths, seed: int, offset: int, req_ids=None):
    """Rejection-sampling verification of a block of draft tokens per request.

    p_target [B, gamma+1, V] float32, p_draft [B, gamma, V] float32,
    draft_tokens [B, gamma] int, lengths [B] or None (all gamma).
    req_ids: request index used in the random-number counter (default 0..B-1).
    """
    B, gamma, _ = np.shape(p_draft)
    u, R = verify_draws(B, gamma, seed, offset, req_ids)
    return verify_given_draws(p_target, p_draft, draft_tokens, lengths, u, R)


def acceptance_probability_exact(pt: float, pd: float) -> float:
    """P(fl32(u * pd) < pt) over the 2**23 equally likely values of u (exact count).

    The closed-form counterpart (for exact real arithmetic) is min(1, pt/pd).
    """
    pt = np.float32(pt)
    pd = np.float32(pd)
    u = ((np.arange(2 ** 23, dtype=np.float64) + 0.5) * 2.0 ** -23).astype(np.float32)
    return float(np.count_nonzero((u * pd).astype(np.float32) < pt)) / 2 ** 23
