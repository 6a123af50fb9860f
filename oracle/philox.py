"""Philox4x32-10 counter-based generator and Gumbel(0,1) rows -- oracle side.

Philox4x32 follows Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
1, 2, 3" (SC'11), section 4: a 10-round Feistel-like network over four 32-bit
counter words and a two-word key; each round takes the 64-bit products of two
counter words with the multipliers M0, M1, swaps and xors the high halves with the
other two words and the round key, and the key advances by the Weyl constants
W0, W1 between rounds.

The Gumbel rows serve the sampling rule of "Depth Exploration for LLM Decoding"
(Appendix C.1, Algorithm 2): one Gumbel(0,1) value per vocabulary entry, shared by
every depth of a slot chain.  Reading adopted here: the row is keyed by
(seed, sequence, absolute target position), so every slot that targets a position
shares the row plain autoregressive sampling uses at that position, which makes the
committed sample stream equal to the AR stream token for token.

Value mapping (both sides implement it from this definition):
  key     = (seed mod 2^32, seed >> 32)
  counter = (v >> 2, target_position, sequence, 0x44455843)
  x       = output word (v & 3)
  U       = ((x >> 9) + 1/2) * 2^-23        -- in (0, 1), exact in fp32
  G       = -log(-log U)
"""
from __future__ import annotations

import numpy as np

MASK32 = np.uint64(0xFFFFFFFF)
M0, M1 = np.uint64(0xD2511F53), np.uint64(0xCD9E8D57)
W0, W1 = np.uint64(0x9E3779B9), np.uint64(0xBB67AE85)
GUMBEL_TAG = 0x44455843


def philox4x32_10(ctr, key):
    """Philox4x32 with 10 rounds.  ctr: four uint32 arrays (broadcastable); key: 2 ints.

    Returns four uint32 numpy arrays.
    """
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & MASK32 for c in ctr)
    c0, c1, c2, c3 = np.broadcast_arrays(c0, c1, c2, c3)
    k0, k1 = np.uint64(key[0] & 0xFFFFFFFF), np.uint64(key[1] & 0xFFFFFFFF)
    for r in range(10):
        p0 = M0 * c0          # < 2^64: exact in uint64
        p1 = M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        if r < 9:
            k0 = (k0 + W0) & MASK32
            k1 = (k1 + W1) & MASK32
    return tuple(c.astype(np.uint32) for c in (c0, c1, c2, c3))


def uniform_open01(x):
    """Map 32-bit words to U in (0, 1): ((x >> 9) + 1/2) * 2^-23."""
    x = np.asarray(x, dtype=np.uint32)
    return ((x >> np.uint32(9)).astype(np.float64) + 0.5) * (2.0 ** -23)


def gumbel_row(seed: int, seq: int, pos: int, vocab: int) -> np.ndarray:
    """G[v] ~ Gumbel(0,1) for v in [0, vocab), keyed by (seed, seq, target position)."""
    nblk = (vocab + 3) // 4
    blk = np.arange(nblk, dtype=np.uint64)
    key = (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    words = philox4x32_10((blk, pos, seq, GUMBEL_TAG), key)
    x = np.stack(words, axis=1).reshape(-1)[:vocab]
    u = uniform_open01(x)
    return -np.log(-np.log(u))
