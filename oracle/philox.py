"""Counter-based random numbers for the dropout mask -- TEST INFRASTRUCTURE ONLY
(imported by tests, the smoke check and the benchmark's CPU leg; never by
the product path, which carries its own implementation of the same
published generator).

The pages state only that the dropout mask is not stored: the forward's
pseudo-random generator state is kept and the mask regenerated in the
backward pass, for O(N) extra memory (page "FlashAttention: Fast and
Memory-Efficient Exact Attention with IO-Awareness", claims on the backward
pass and dropout).  They name no generator.  This module implements
Philox4x32-10 from its published definition (J. K. Salmon, M. A. Moraes,
R. O. Dror, D. E. Shaw, "Parallel random numbers: as easy as 1, 2, 3",
SC'11): a 4 x 32-bit counter and a 2 x 32-bit key; each of ten rounds
multiplies counter words 0 and 2 by two fixed odd constants, forms the new
counter from the high and low halves of the products crossed with words 1
and 3 and the key, and advances the key by two Weyl constants.

Element mapping (the reading used by both sides): for head index bh = b*H+h,
query row i, key column j (positions within the head or packed sequence),
the counter is (j // 16, i, bh, offset) and the key (seed mod 2^32,
seed >> 32); byte (j % 16) of the 16 output bytes (word (j % 16) // 4, bits
8*(j % 4) ..) is a uniform integer u in [0, 256); the element is kept iff
u >= p8, where p8 = round(p_drop * 256) in [0, 255].  A kept probability is
scaled by 1 / (1 - p8 / 256) (inverted dropout).
"""

import numpy as np

M0 = np.uint64(0xD2511F53)
M1 = np.uint64(0xCD9E8D57)
W0 = np.uint32(0x9E3779B9)
W1 = np.uint32(0xBB67AE85)
MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32-10 on arrays of counters (broadcast): returns 4 uint32 arrays."""
    c = [np.asarray(x, dtype=np.uint64) & MASK32 for x in (c0, c1, c2, c3)]
    c = list(np.broadcast_arrays(*c))
    k0 = np.uint64(int(k0) & 0xFFFFFFFF)
    k1 = np.uint64(int(k1) & 0xFFFFFFFF)
    for r in range(10):
        if r > 0:
            k0 = (k0 + np.uint64(W0)) & MASK32
            k1 = (k1 + np.uint64(W1)) & MASK32
        p0 = M0 * c[0]          # < 2^64: 32 x 32-bit product in uint64
        p1 = M1 * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return [x.astype(np.uint32) for x in c]


def dropout_p8(p_drop):
    """The dropout probability in steps of 1/256, as both sides use it."""
    if not 0.0 <= p_drop < 1.0:
        raise ValueError("p_drop must be in [0, 1)")
    return min(255, int(round(p_drop * 256)))


def dropout_keep(seed, offset, p8, bh, rows, cols):
    """Boolean [len(rows), len(cols)]: which (i, j) of head bh are kept."""
    rows = np.asarray(rows, dtype=np.uint64)[:, None]
    cols = np.asarray(cols, dtype=np.uint64)[None, :]
    w = philox4x32_10(cols // np.uint64(16), rows, np.uint64(bh), np.uint64(offset),
                      int(seed) & 0xFFFFFFFF, (int(seed) >> 32) & 0xFFFFFFFF)
    jj = (cols % np.uint64(16)).astype(np.int64)
    word = np.choose(np.broadcast_to(jj // 4, w[0].shape), w)
    u = (word >> (8 * np.broadcast_to(jj % 4, w[0].shape)).astype(np.uint32)) & np.uint32(0xFF)
    return u >= p8
