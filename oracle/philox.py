"""Philox-4x32-10 counter-based generator and the uniforms of the accept step.

Definition (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
1, 2, 3", SC'11, section 4 "Philox"): a 128-bit counter (c0, c1, c2, c3) and a
64-bit key (k0, k1) go through 10 rounds.  One round takes the two 32x32 -> 64
bit products M0 * c0 and M1 * c2 and forms

    (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0))

with M0 = 0xD2511F53 and M1 = 0xCD9E8D57.  Between rounds the key advances by
the Weyl constants (0x9E3779B9, 0xBB67AE85) modulo 2^32; the first round uses
the key as given.

Uniforms [reading: the pages fix no generator; the accept rule only needs
u in [0, 1)].  Element i of the stream (seed, subsequence) at offset o is
word (o + i) % 4 of Philox(counter = (b mod 2^32, b >> 32, s mod 2^32, s >> 32),
key = (seed mod 2^32, seed >> 32)) with b = (o + i) // 4 and s the
subsequence; the word x becomes u = (x >> 8) * 2^-24, exact in fp32.
"""

import numpy as np

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
MASK32 = 0xFFFFFFFF


def philox4x32_10(counter, key):
    """Four uint32 outputs (Python ints) for a 4-word counter and 2-word key."""
    c0, c1, c2, c3 = (int(v) & MASK32 for v in counter)
    k0, k1 = (int(v) & MASK32 for v in key)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + W0) & MASK32
            k1 = (k1 + W1) & MASK32
        p0 = M0 * c0
        p1 = M1 * c2
        c0, c1, c2, c3 = ((p1 >> 32) ^ c1 ^ k0, p1 & MASK32,
                          (p0 >> 32) ^ c3 ^ k1, p0 & MASK32)
    return c0, c1, c2, c3


def uniforms(seed, subsequence, offset, n):
    """fp32 [n] uniforms in [0, 1) of stream (seed, subsequence) from ``offset``."""
    seed, subsequence, offset = int(seed), int(subsequence), int(offset)
    key = (seed & MASK32, (seed >> 32) & MASK32)
    out = np.empty(n, dtype=np.float32)
    cached_block, words = None, None
    for i in range(n):
        idx = offset + i
        block = idx // 4
        if block != cached_block:
            ctr = (block & MASK32, (block >> 32) & MASK32,
                   subsequence & MASK32, (subsequence >> 32) & MASK32)
            words, cached_block = philox4x32_10(ctr, key), block
        out[i] = np.float32((words[idx % 4] >> 8) * 2.0 ** -24)
    return out
