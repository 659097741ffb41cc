"""Sampling on a reduced draft vocabulary (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources:
  * "DSpark implementation and evaluation" §5: the draft computes its logits
    on a small vocabulary and scatters them into the target vocabulary's
    positions (every other position -inf) through an index table, so a
    sampled draft entry d stands for target token d2t[d] ("index" mode);
  * "xserv/docs/25-speculative-methods-comparison.md" §3.2 (EAGLE-3): the
    draft predicts a draft-vocabulary id and the table gives an offset,
    real_id = draft_id + d2t[draft_id] ("offset" mode).

Readings:
  * the whole Markov chain runs on draft ids: base logits [B, N, V_draft],
    markov_w1 / markov_w2 [V_draft, r], the anchor and every fed-back token are
    draft ids (the embedding table is the draft's);
  * Gumbel-max over the scattered target-size buffer (-inf off the draft
    positions) draws from the same distribution as Gumbel-max over the draft
    entries; the noise is indexed by draft id and ties go to the lowest draft
    id;
  * only the returned tokens are mapped to target ids; a mapped id outside
    [0, V_target) is returned as -1 (the GPU also raises a flag).
"""
from __future__ import annotations

import numpy as np

from .draft import markov_sample

MODE_INDEX, MODE_OFFSET = 0, 1


def map_to_target(draft_ids: np.ndarray, d2t: np.ndarray, mode: int, V_target: int) -> np.ndarray:
    """Target-vocabulary ids of draft ids: d2t[d] (index mode) or d + d2t[d] (offset mode)."""
    d = np.asarray(draft_ids, dtype=np.int64)
    table = np.asarray(d2t, dtype=np.int64)
    t = table[d] if mode == MODE_INDEX else d + table[d]
    return np.where((t >= 0) & (t < V_target), t, -1)


def markov_sample_reduced(base_logits, anchor, w1, w2, temperature, seed: int, offset: int,
                          d2t, mode: int, V_target: int, req_ids=None, forced_draft_tokens=None):
    """Returns (target tokens [Bs, N], draft tokens [Bs, N], gap, lse) -- gap and lse as in
    ``markov_sample`` (computed on the draft vocabulary).  forced_draft_tokens: teacher
    forcing with a sequence of draft ids (``markov_sample``'s forced_tokens)."""
    draft, gap, lse = markov_sample(base_logits, anchor, w1, w2, temperature, seed, offset, req_ids,
                                    forced_tokens=forced_draft_tokens)
    return map_to_target(draft, d2t, mode, V_target), draft, gap, lse
