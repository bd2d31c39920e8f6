"""Philox4x32-10, the counter-based generator behind the dropout contract.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: the library has its
own implementation and shares nothing with this one.

The generator is the one of Salmon, Moraes, Dror and Shaw, "Parallel Random
Numbers: As Easy as 1, 2, 3" (SC 2011), Philox with four 32-bit words and
ten rounds.  A 128-bit counter (c0, c1, c2, c3) and a 64-bit key (k0, k1)
map to four 32-bit outputs.  Each round takes the two 64-bit products
M0 * c0 and M1 * c2 and forms the next counter as
    (hi(M1 c2) ^ c1 ^ k0,  lo(M1 c2),  hi(M0 c0) ^ c3 ^ k1,  lo(M0 c0)),
and between rounds the key words grow by the Weyl constants W0 and W1
(mod 2^32).  The constants are the paper's for this variant.  The
known-answer vectors distributed with the paper's Random123 library pin
this code (tests/golden/philox4x32_10_kat.txt).
"""
from __future__ import annotations

import numpy as np

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
_MASK = np.uint64(0xFFFFFFFF)


def philox4x32_10(counter, key):
    """Vectorised Philox4x32-10.

    counter: four integer arrays (or scalars) that broadcast together, each
    holding 32-bit values; key: two 32-bit integers.  Returns the four output
    words as uint64 arrays holding 32-bit values.
    """
    c = [np.asarray(x, dtype=np.uint64) & _MASK for x in counter]
    c = list(np.broadcast_arrays(*c))
    k0, k1 = int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF
    for r in range(10):
        if r:
            k0 = (k0 + W0) & 0xFFFFFFFF
            k1 = (k1 + W1) & 0xFFFFFFFF
        p0 = np.uint64(M0) * c[0]  # < 2^64: both factors are below 2^32
        p1 = np.uint64(M1) * c[2]
        c = [(p1 >> np.uint64(32)) ^ c[1] ^ np.uint64(k0), p1 & _MASK,
             (p0 >> np.uint64(32)) ^ c[3] ^ np.uint64(k1), p0 & _MASK]
    return c
