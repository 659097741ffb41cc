"""Confidence-scheduled admission of draft tokens (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "Speculative decoding: from zero to DSpark" (bittide.aicompass.dev)
  §6 -- per-position conditional acceptance probabilities are chained into
       survival probabilities (monotone non-increasing within a request);
       all candidate extensions of all requests are pooled, sorted by
       survival and admitted from the top; the verify length is chosen to
       maximise expected tokens per batch x SPS(batch size).  Admission of
       token k must not depend on the value of token k (non-anticipation).
  §7 -- the SPS curve is jagged at kernel-tile boundaries, so the search does
       not stop early; the capacity K may be fixed two steps ahead and the K
       slots filled at the last moment by sorting the live candidates.

Readings:
  * survival s_{b,0} = c_{b,0}, s_{b,k} = fl32(s_{b,k-1} * c_{b,k}); c is
    clamped to [0, 1] (NaN -> 0) and the clamp raises a flag;
  * candidates sort by (s descending, then flat index b*N+k ascending): ties
    inside a request keep position order, so every admitted set is
    prefix-closed per request;
  * expected tokens of a batch that admits the top K candidates is
    B + sum of their survivals (every request also gets one target token,
    the correction or the bonus); it is evaluated in fixed point:
    E(K) = B * 2**32 + sum_{j<K} floor(s_(j) * 2**32), exact in 64 bits;
  * the SPS table is indexed by K (entry K-1 is batch size K);
    f(K) = float64(E(K)) * SPS[K-1]; K* = the smallest K in
    [1, min(B*N, S)] attaining the maximum, every K evaluated;
  * K_in >= 0 fixes K (clamped to B*N) and skips the search (the
    two-steps-ahead mode of §7).
"""
from __future__ import annotations

import numpy as np

TWO32 = float(2 ** 32)


def survival_chain(cond_accept: np.ndarray):
    """Chain rule: s_{b,k} = prod_{j<=k} c_{b,j}, each product rounded to float32.

    Returns (survival [B, N] float32, clamped flag).
    """
    c = np.asarray(cond_accept, dtype=np.float32)
    bad = ~((c >= 0) & (c <= 1))          # also catches NaN
    cc = np.where(np.isnan(c), np.float32(0), np.clip(c, np.float32(0), np.float32(1)))
    s = np.empty_like(cc)
    s[:, 0] = cc[:, 0]
    for k in range(1, cc.shape[1]):
        s[:, k] = (s[:, k - 1] * cc[:, k]).astype(np.float32)
    return s, bool(bad.any())


def schedule(cond_accept: np.ndarray, sps: np.ndarray | None, K_in: int):
    """Admission of the top-K candidates by survival.

    Returns dict: survival [B,N] float32, K (int), lengths [B] int64,
    selected [B*N] int64 (flat b*N+k of the admitted candidates in sort order,
    then -1), order [B*N] (full sort order), clamped (bool).
    """
    s, clamped = survival_chain(cond_accept)
    B, N = s.shape
    n = B * N
    flat = s.reshape(-1)
    # sort by (s descending, flat index ascending); lexsort's last key is primary
    order = np.lexsort((np.arange(n), -flat.astype(np.float64)))
    if K_in >= 0:
        K = min(int(K_in), n)
    else:
        S = len(sps)
        Kmax = min(n, S)
        q = [int(np.floor(float(flat[j]) * TWO32)) for j in order[:Kmax]]
        E = B * 2 ** 32
        best_f, K = -np.inf, 1
        for k in range(1, Kmax + 1):          # every K: no early stop (§7)
            E += q[k - 1]
            f = float(E) * float(sps[k - 1])
            if f > best_f:                     # strict: ties keep the smallest K
                best_f, K = f, k
    selected = np.full(n, -1, dtype=np.int64)
    selected[:K] = order[:K]
    lengths = np.zeros(B, dtype=np.int64)
    for j in order[:K]:
        lengths[j // N] += 1
    return {"survival": s, "K": K, "lengths": lengths, "selected": selected,
            "order": order, "clamped": clamped}
