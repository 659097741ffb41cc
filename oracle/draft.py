"""Draft step of DSpark (oracle side): base logits and sequential Markov sampling.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "DSpark implementation and evaluation" (ggaaooppeenngg.github.io)
  §2.2 Sequential Markov Sampling -- the backbone's N hidden states go through
       the draft LM head once, giving base logits [B, N, V]; then for
       i = 0..N-1 in order the previous token (the anchor for i = 0) is
       embedded by markov_w1, projected to a vocabulary-sized bias by
       markov_w2, added to base_logits[:, i], and a token is Gumbel-sampled
       and becomes the next step's previous token.
  §3   Markov Head structure -- markov_w1 is an Embedding(V, r) and markov_w2
       a bias-free r -> V linear; both stored here as [V, r] row-major.
  §4   the draft step = one parallel forward + the sequential loop.
"Speculative decoding: from zero to DSpark" §4 describes the same head as a
learned V x V bigram table factored at low rank.

Readings where the pages are silent:
  * the bias is added to the base logits BEFORE temperature scaling (the
    page passes base + bias to the Gumbel sampler);
  * temperature T > 0 divides (base + bias); T = 0 means greedy argmax of
    base + bias, with no noise;
  * Gumbel-max: x = argmax_v (z_v + g_v), ties to the lowest index;
  * the draft vocabulary equals the target vocabulary (no d2t map).
"""
from __future__ import annotations

import numpy as np

from .philox import draft_gumbel


def draft_logits(hidden: np.ndarray, lm_head: np.ndarray) -> np.ndarray:
    """Base logits L[m, v] = sum_h hidden[m, h] * lm_head[v, h], in float64.

    "DSpark implementation and evaluation" §2.2 (compute_draft_logits over all N
    positions at once) and §4 step 2.  Inputs hold the exact stored values
    (bf16 or fp32); the product is taken in float64 by numpy's matmul.
    """
    return np.asarray(hidden, dtype=np.float64) @ np.asarray(lm_head, dtype=np.float64).T


def markov_bias(prev: np.ndarray, w1: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """markov_bias(markov_embed(prev)) = w2 @ w1[prev] for each request: [len(prev), V] float64.

    "DSpark implementation and evaluation" §3: markov_w1 is an embedding lookup
    (prev -> [r]) and markov_w2 a bias-free linear r -> V.
    """
    emb = np.asarray(w1, dtype=np.float64)[np.asarray(prev, dtype=np.int64)]   # [b, r]
    return emb @ np.asarray(w2, dtype=np.float64).T                             # [b, V]


def markov_sample_given_noise(base_logits, anchor, w1, w2, temperature, gumbel, forced_tokens=None):
    """The sequential loop with the Gumbel noise supplied.

    gumbel(i, rows) -> [len(rows), V] float64 noise of step i for the local
    request rows `rows` (only rows with T > 0 are asked for).

    forced_tokens [Bs, N] (optional): teacher forcing.  Step i + 1 then embeds
    forced_tokens[:, i] as its previous token instead of this loop's own token
    of step i.  Each step is still the step of §2.2 (bias of the previous
    token, add, temperature, Gumbel-max); only the history it conditions on is
    supplied, so that another implementation's token sequence can be checked
    position by position without one near tie changing every later step.

    Returns (tokens [Bs, N] int64, gap [Bs, N] float64, lse [Bs, N] float64):
      gap = (largest - second largest) of the perturbed values at each step,
      lse = log-sum-exp over v of z = (base + bias) / T  (T = 0: of base + bias).
    """
    L = np.asarray(base_logits, dtype=np.float64)
    Bs, N, V = L.shape
    T = np.asarray(temperature, dtype=np.float64).reshape(Bs)
    prev = np.asarray(anchor, dtype=np.int64).reshape(Bs).copy()
    tokens = np.empty((Bs, N), dtype=np.int64)
    gap = np.empty((Bs, N), dtype=np.float64)
    lse = np.empty((Bs, N), dtype=np.float64)
    rows = np.arange(Bs)
    hot = T > 0
    for i in range(N):
        logits = L[:, i, :] + markov_bias(prev, w1, w2)           # base_logits[:, i] + bias
        z = logits / np.where(hot, T, 1.0)[:, None]
        y = z.copy()
        if hot.any():
            y[hot] += gumbel(i, rows[hot])
        x = np.argmax(y, axis=1)                                  # first maximum = lowest index
        top1 = y[rows, x]
        y[rows, x] = -np.inf
        gap[:, i] = top1 - y.max(axis=1)
        m = z.max(axis=1)
        lse[:, i] = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
        tokens[:, i] = x
        if forced_tokens is None:
            prev = x                                               # feeds the next step
        else:
            prev = np.asarray(forced_tokens, dtype=np.int64)[:, i].copy()
    return tokens, gap, lse


def markov_sample(base_logits, anchor, w1, w2, temperature, seed: int, offset: int,
                  req_ids=None, forced_tokens=None):
    """Sequential Markov-biased Gumbel-max sampling of N draft tokens per request.

    "DSpark implementation and evaluation" §2.2 (the sequential loop) and §3.

    base_logits [Bs, N, V]: base logits of the requests req_ids (default 0..Bs-1);
    req_ids give the request index b used in the random-number counter, so a
    subset of a large batch can be checked alone.  anchor, temperature: [Bs].
    The Gumbel noise of step i, request b, token v is ``philox.draft_gumbel``:
    entries in groups of 16 (G = v >> 4, k = v & 15); the group word is word
    G & 3 of the stream-0 counter (G >> 2, b, i, offset) and gives the position
    of the group's largest variate and the group's smallest exponential; every
    other entry adds its own exponential from word k & 3 of the stream-3 counter
    ((G << 2) | (k >> 2), b, i, offset); g = -log(E).
    forced_tokens: teacher forcing, as in ``markov_sample_given_noise``.
    """
    L = np.asarray(base_logits)
    req = np.arange(L.shape[0]) if req_ids is None else np.asarray(req_ids)
    V = L.shape[2]

    def gumbel(i, rows):
        return draft_gumbel(seed, offset, req[rows], i, V)

    return markov_sample_given_noise(base_logits, anchor, w1, w2, temperature, gumbel, forced_tokens)
