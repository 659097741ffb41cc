"""Confidence head with per-position calibration (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "Speculative decoding: from zero to DSpark" (bittide.aicompass.dev) §6:
the survival probability of each draft token comes from a confidence head -- a
linear projection of the backbone's hidden state together with the Markov
embedding -- that predicts each position's conditional acceptance probability;
the chain rule turns those into survival probabilities (``survival_chain``),
and each position is calibrated with temperature scaling.

Readings (the page gives the structure, not the formula):
  * the projection acts on the concatenation [h_{b,i}; E_{b,i}] with one weight
    vector split as (w_h over the H hidden features, w_e over the r Markov
    features) and a scalar bias beta, giving a logit;
  * E_{b,i} = markov_w1[prev] is the embedding the Markov head uses at step i:
    prev = the anchor token for i = 0, the draft token x_{b,i-1} after;
  * the logit is squashed by a sigmoid into a probability; temperature scaling
    divides the logit by the position's temperature tau_i > 0 before it:
        c_{b,i} = 1 / (1 + exp(-(w_h . h_{b,i} + w_e . E_{b,i} + beta) / tau_i)).
"""
from __future__ import annotations

import numpy as np


def confidence(hidden: np.ndarray, w1: np.ndarray, anchor: np.ndarray, draft_tokens: np.ndarray,
               w_h: np.ndarray, w_e: np.ndarray, beta: float, tau: np.ndarray) -> np.ndarray:
    """hidden [B*N, H] (row b*N + i), w1 [V, r], anchor [B], draft_tokens [B, N], w_h [H], w_e [r],
    tau [N] -> conditional acceptance probabilities c [B, N] (float64)."""
    x = np.asarray(draft_tokens, dtype=np.int64)
    B, N = x.shape
    h = np.asarray(hidden, dtype=np.float64).reshape(B, N, -1)
    W1 = np.asarray(w1, dtype=np.float64)
    prev = np.concatenate([np.asarray(anchor, dtype=np.int64)[:, None], x[:, :-1]], axis=1)   # [B, N]
    E = W1[prev]                                                                                # [B, N, r]
    logit = h @ np.asarray(w_h, dtype=np.float64) + E @ np.asarray(w_e, dtype=np.float64) + float(beta)
    z = logit / np.asarray(tau, dtype=np.float64)[None, :]
    return 1.0 / (1.0 + np.exp(-z))
