"""Philox4x32-10 in plain Python, written from its published definition.

Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
(SC'11): a 4x32-bit counter and a 2x32-bit key; each of 10 rounds multiplies
words 0 and 2 by fixed 32-bit constants, keeps both halves of the products,
and mixes the high halves with the other two words and the round key; the key
is bumped by two Weyl constants between rounds.

Used by the tests to check the GPU's block visiting order, which the selector
draws from this generator (the shuffled block order of The Secret GPU Kernel
Behind DeepSeek V4.1 Flash, video transcript 3:30 and 4:55-5:10).
"""

MASK = 0xFFFFFFFF
M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85


def philox4x32_10(ctr, key):
    c0, c1, c2, c3 = (int(v) & MASK for v in ctr)
    k0, k1 = (int(v) & MASK for v in key)
    for _ in range(10):
        p0 = M0 * c0
        p1 = M1 * c2
        hi0, lo0 = (p0 >> 32) & MASK, p0 & MASK
        hi1, lo1 = (p1 >> 32) & MASK, p1 & MASK
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = (k0 + W0) & MASK
        k1 = (k1 + W1) & MASK
    return c0, c1, c2, c3
