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
  stream 0 = draft noise, high halves (b = request, i = draft step)
  stream 3 = draft noise, low halves  (same counters)
             element v takes 16 bits from each stream, from counter j = v >> 3:
             word (v & 7) >> 1, bits 0-15 for even v and 16-31 for odd v;
             its 32-bit word is (high half << 16) | low half
  (the split lets a sampler rule an element out from its high half alone,
  since u, and so g, is increasing in the word)
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


def draft_halfword(seed: int, offset: int, b, i, v, stream: int) -> np.ndarray:
    """16-bit piece of element v's draft word from `stream` (0: high half, 3: low half)."""
    v = np.asarray(v, dtype=np.uint64)
    words = philox_words(seed, offset, v >> np.uint64(3), b, stream, i)
    sel = ((v & np.uint64(7)) >> np.uint64(1)).astype(np.int64)
    w = np.where(sel == 0, words[0], np.where(sel == 1, words[1],
                 np.where(sel == 2, words[2], words[3])))
    shift = (v & np.uint64(1)) * np.uint64(16)
    return (w >> shift) & np.uint64(0xFFFF)


def draft_word(seed: int, offset: int, b, i, v) -> np.ndarray:
    """32-bit draft-noise word of element v: (high half << 16) | low half."""
    hi = draft_halfword(seed, offset, b, i, v, STREAM_GUMBEL)
    lo = draft_halfword(seed, offset, b, i, v, STREAM_GUMBEL_LO)
    return (hi << np.uint64(16)) | lo


def draft_gumbel(seed: int, offset: int, b, i, V: int) -> np.ndarray:
    """Gumbel noise g[b, v] (float64) of draft step i for requests b (array) over v in [0, V)."""
    b = np.asarray(b, dtype=np.uint64).reshape(-1, 1)
    v = np.arange(V, dtype=np.uint64).reshape(1, -1)
    return gumbel_from_word(draft_word(seed, offset, b, i, v))
