"""Philox4x32-10 and the random variates the method draws from it (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The generator is the counter-based Philox4x32 with 10 rounds from Salmon,
Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11):
a 128-bit counter (c0, c1, c2, c3) and a 64-bit key (k0, k1).  Each round
multiplies c0 by 0xD2511F53 and c2 by 0xCD9E8D57 (full 64-bit products),
then outputs
    (hi(c2*M1) ^ c1 ^ k0,  lo(c2*M1),  hi(c0*M0) ^ c3 ^ k1,  lo(c0*M0))
and the key is bumped by the Weyl constants (0x9E3779B9, 0xBB67AE85)
between rounds.

The pages only say that drafting samples with Gumbel noise and that
verification uses a seeded uniform ("DSpark implementation and evaluation"
§2.2 and §5).  The counter layout below is this library's reading:

  key      = (lo32(seed), hi32(seed))
  counter  = (j, b, (stream << 16) | i, offset)       offset < 2**32
  stream 0 = draft noise, group words (b = request, i = draft step)
  stream 3 = draft noise, element words (same b, i)
             entries come in groups of 16 (G = v >> 4, position k = v & 15);
             the group word is word G & 3 of counter j = G >> 2 of stream 0:
             its bits 0-3 give the position p of the group's largest variate,
             its uniform u0 the group's smallest exponential E_min = -log(u0) / 16;
             entry k != p takes word k & 3 of counter j = (G << 2) | (k >> 2)
             of stream 3 and E_k = E_min - log(u_k); E_p = E_min; g = -log(E).
             The smallest of 16 independent Exp(1) variates is Exp(16)
             distributed, its position uniform, and the others exceed it by
             independent Exp(1) amounts, so the 16 E's are independent Exp(1)
             and the g's independent standard Gumbels; -log(E_min), which is
             u0's Gumbel variate + log 16, bounds every g of the group, so a
             sampler can rule a whole group out from one word
  stream 1 = verify accept uniform   (i = draft position k, j = 0, word 0)
  stream 2 = verify resample         (i = position, j = 0, words 0 and 1)
  stream 4 = from-logits resample    (i = position, j = v >> 2, word v & 3 of element v)

Uniform: u = ((w >> 9) + 1/2) * 2**-23, which lies in [2**-24, 1 - 2**-24]
and is exactly representable in float32.  Gumbel: g = -log(-log(u)).
"""
from __future__ import annotations

import numpy as np

M0 = np.uint64(0xD2511F53)
M1 = np.uint64(0xCD9E8D57)
W0 = np.uint64(0x9E3779B9)
W1 = np.uint64(0xBB67AE85)
MASK = np.uint64(0xFFFFFFFF)
S32 = np.uint64(32)

STREAM_GUMBEL = 0
STREAM_ACCEPT = 1
STREAM_RESAMPLE = 2
STREAM_GUMBEL_LO = 3
STREAM_RESIDUAL = 4          # Gumbel noise of the from-logits resample draw


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32-10 on (broadcastable) arrays of 32-bit values held in uint64.

    Returns the four 32-bit output words as uint64 arrays.
    """
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & MASK for c in (c0, c1, c2, c3))
    k0 = np.asarray(k0, dtype=np.uint64) & MASK
    k1 = np.asarray(k1, dtype=np.uint64) & MASK
    for _ in range(10):
        p0 = c0 * M0          # < 2**64: exact
        p1 = c2 * M1
        c0, c1, c2, c3 = ((p1 >> S32) ^ c1 ^ k0,
                          p1 & MASK,
                          (p0 >> S32) ^ c3 ^ k1,
                          p0 & MASK)
        k0 = (k0 + W0) & MASK
        k1 = (k1 + W1) & MASK
    return c0, c1, c2, c3


def _key(seed: int):
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return np.uint64(seed & 0xFFFFFFFF), np.uint64(seed >> 32)


def philox_words(seed: int, offset: int, j, b, stream: int, i):
    """The four output words for counter (j, b, (stream << 16) | i, offset)."""
    if not 0 <= int(offset) < 2 ** 32:
        raise ValueError("offset must be below 2**32")
    k0, k1 = _key(seed)
    c2 = (np.uint64(stream) << np.uint64(16)) | np.asarray(i, dtype=np.uint64)
    return philox4x32_10(j, b, c2, np.uint64(offset), k0, k1)


def uniform_from_word(w) -> np.ndarray:
    """u = ((w >> 9) + 0.5) * 2**-23 as float64 (exactly a float32 value)."""
    w = np.asarray(w, dtype=np.uint64)
    return ((w >> np.uint64(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def gumbel_from_word(w) -> np.ndarray:
    """Standard Gumbel variate g = -log(-log(u)) in float64."""
    u = uniform_from_word(w)
    return -np.log(-np.log(u))


GROUP = 16                   # draft-noise entries per group word


def _select_word(words, idx):
    """words: the 4 output arrays of philox_words; idx: which word (0..3), broadcastable."""
    idx = np.asarray(idx)
    return np.where(idx == 0, words[0], np.where(idx == 1, words[1], np.where(idx == 2, words[2], words[3])))


def draft_group_words(seed: int, offset: int, b, i, G) -> np.ndarray:
    """Group word of draft-noise group G: word G & 3 of counter (G >> 2, b, (0 << 16) | i, offset)."""
    G = np.asarray(G, dtype=np.uint64)
    words = philox_words(seed, offset, G >> np.uint64(2), b, STREAM_GUMBEL, i)
    return _select_word(words, (G & np.uint64(3)).astype(np.int64))


def draft_gumbel(seed: int, offset: int, b, i, V: int) -> np.ndarray:
    """Gumbel noise g[b, v] (float64) of draft step i for requests b (array) over v in [0, V).

    Groups of 16 entries: the group word gives the position p of the group's largest variate
    (its bits 0-3) and the group's smallest exponential E_min = -log(u0) / 16; every other
    entry k adds its own exponential, E_k = E_min - log(u_k), from word k & 3 of the stream-3
    counter (G << 2) | (k >> 2); g = -log(E).
    """
    b = np.asarray(b, dtype=np.uint64).reshape(-1, 1)
    n_groups = (V + GROUP - 1) // GROUP
    G = np.arange(n_groups, dtype=np.uint64).reshape(1, -1)
    W = draft_group_words(seed, offset, b, i, G)                           # [nb, n_groups]
    p = (W & np.uint64(15)).astype(np.int64)
    e_min = -np.log(uniform_from_word(W)) / GROUP
    v = np.arange(n_groups * GROUP, dtype=np.uint64).reshape(1, -1)
    k = v & np.uint64(15)
    Gv = (v >> np.uint64(4)).astype(np.int64).ravel()
    ew = _select_word(philox_words(seed, offset, ((v >> np.uint64(4)) << np.uint64(2)) | (k >> np.uint64(2)),
                                   b, STREAM_GUMBEL_LO, i), (k & np.uint64(3)).astype(np.int64))
    E = e_min[:, Gv] - np.log(uniform_from_word(ew))
    E = np.where(k.astype(np.int64) == p[:, Gv], e_min[:, Gv], E)
    return -np.log(E)[:, :V]
