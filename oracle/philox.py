"""Philox4x32-10 counter-based generator, written from its published definition.

Reference: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel Random
Numbers: As Easy as 1, 2, 3", SC'11, section 4 (the Philox S-box: two 32x32->64
multiplies per round, a Weyl sequence for the round keys, 10 rounds).

Test infrastructure only (see oracle/__init__.py).

Per-vocabulary-entry uniforms used by the draw (the sampled frame of "Qwen3-TTS:
Run the 1.7B Depth Loop as One Persistent Kernel on Hopper", section "How it
works": each draw reads the row's seed and offset): entry v of row r at
offset o reads word (v mod 4) of Philox4x32-10 with
key = (seed low 32 bits, seed high 32 bits) and
counter = (v div 4, r, o low 32 bits, o high 32 bits),
mapped to ((word >> 9) + 0.5) * 2^-23, which is exact in float32 (24
significant bits) and lies strictly inside (0, 1): from 2^-24 to 1 - 2^-24.
(With 24 kept bits the top value 2^24 - 0.5 would need 25 bits and round to
exactly 1, making -log(-log u) infinite.)
"""
from __future__ import annotations

import numpy as np

M0 = 0xD2511F53   # multiplier applied to counter word 0
M1 = 0xCD9E8D57   # multiplier applied to counter word 2
W0 = 0x9E3779B9   # key increment for key word 0 (golden ratio)
W1 = 0xBB67AE85   # key increment for key word 1 (sqrt(3) - 1)
ROUNDS = 10
_M32 = np.uint64(0xFFFFFFFF)


def philox4x32(ctr, key, rounds: int = ROUNDS):
    """Philox4x32 with ``rounds`` rounds.

    ``ctr``: 4 arrays (or ints) of 32-bit counter words; ``key``: 2 arrays (or
    ints) of 32-bit key words; all broadcast together. Returns 4 uint32 arrays.

    One round maps (c0, c1, c2, c3) with key (k0, k1) to
    (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0)),
    and the key advances by (W0, W1) between rounds.
    """
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & _M32 for c in ctr)
    k0, k1 = (np.asarray(k, dtype=np.uint64) & _M32 for k in key)
    c0, c1, c2, c3, k0, k1 = np.broadcast_arrays(c0, c1, c2, c3, k0, k1)
    c0, c1, c2, c3, k0, k1 = (a.copy() for a in (c0, c1, c2, c3, k0, k1))
    for i in range(rounds):
        p0 = c0 * np.uint64(M0)          # 32x32 -> 64 bits, exact in uint64
        p1 = c2 * np.uint64(M1)
        n0 = (p1 >> np.uint64(32)) ^ c1 ^ k0
        n1 = p1 & _M32
        n2 = (p0 >> np.uint64(32)) ^ c3 ^ k1
        n3 = p0 & _M32
        c0, c1, c2, c3 = n0, n1, n2, n3
        if i + 1 < rounds:
            k0 = (k0 + np.uint64(W0)) & _M32
            k1 = (k1 + np.uint64(W1)) & _M32
    return tuple(a.astype(np.uint32) for a in (c0, c1, c2, c3))


def uniform_from_word(word) -> np.ndarray:
    """Map 32-bit words to float32 uniforms ((word >> 9) + 0.5) * 2^-23 in (0, 1).

    The result is exact in float32: at most 24 significant bits."""
    w = np.asarray(word, dtype=np.uint32)
    return ((w >> np.uint32(9)).astype(np.float32) + np.float32(0.5)) * np.float32(2.0 ** -23)


def vocab_words(seed: int, row: int, offset: int, vocab: int) -> np.ndarray:
    """The 32-bit Philox word assigned to each vocabulary entry of one draw."""
    v = np.arange(vocab, dtype=np.uint64)
    seed = int(seed) & ((1 << 64) - 1)
    offset = int(offset) & ((1 << 64) - 1)
    key = (seed & 0xFFFFFFFF, seed >> 32)
    ctr = (v >> np.uint64(2), row, offset & 0xFFFFFFFF, offset >> 32)
    words = np.stack(philox4x32(ctr, key), axis=0)          # [4][vocab]
    return words[(v & np.uint64(3)).astype(np.int64), np.arange(vocab)]


def vocab_uniforms(seed: int, row: int, offset: int, vocab: int) -> np.ndarray:
    """float32 uniforms u_v in (0, 1), one per vocabulary entry, for one draw."""
    return uniform_from_word(vocab_words(seed, row, offset, vocab))
