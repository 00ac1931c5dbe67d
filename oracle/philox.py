"""Philox4x32-10 counter-based generator (oracle side; test infrastructure only).

Written from the published definition: J. K. Salmon, M. A. Moraes, R. O. Dror,
D. E. Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11, §3 (the
Philox S-box: two 32x32->64 multiplications per round, a Weyl key schedule).

One round maps the counter (c0, c1, c2, c3) under round key (k0, k1) to

    (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0))

and the key advances by the Weyl constants between rounds.  Ten rounds.

The dropout of the lesson ("第 7 课：序列并行 SP", answer to Q1) only requires
that every rank uses the same seed so that masks agree and cover the whole
tensor; the choice of a counter-based generator keyed on the global element
index is this build's reading of that requirement.
"""
import numpy as np

MUL0 = 0xD2511F53
MUL1 = 0xCD9E8D57
WEYL0 = 0x9E3779B9
WEYL1 = 0xBB67AE85
ROUNDS = 10

_LO32 = np.uint64(0xFFFFFFFF)
_SH32 = np.uint64(32)


def philox4x32(counter, key, rounds=ROUNDS):
    """Apply Philox4x32-R to arrays of counters.

    counter: sequence of four uint32-valued arrays (c0, c1, c2, c3), all of one
             shape.  key: two uint32 ints (k0, k1).
    Returns a list of four uint32 arrays.
    """
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & _LO32 for c in counter)
    k0 = np.uint64(int(key[0]) & 0xFFFFFFFF)
    k1 = np.uint64(int(key[1]) & 0xFFFFFFFF)
    m0 = np.uint64(MUL0)
    m1 = np.uint64(MUL1)
    for _ in range(rounds):
        prod0 = m0 * c0           # < 2**64: exact in uint64
        prod1 = m1 * c2
        hi0, lo0 = prod0 >> _SH32, prod0 & _LO32
        hi1, lo1 = prod1 >> _SH32, prod1 & _LO32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = (k0 + np.uint64(WEYL0)) & _LO32
        k1 = (k1 + np.uint64(WEYL1)) & _LO32
    return [c.astype(np.uint32) for c in (c0, c1, c2, c3)]


def element_uniforms(seed, offset, elem_index):
    """One uint32 draw per tensor element, keyed on its global linear index.

    Reading (the pages fix no generator): element ``i`` of the full (b, s, h)
    tensor takes word ``i mod 4`` of Philox4x32-10 with
        key     = (seed mod 2**32, seed >> 32)
        counter = (q mod 2**32, q >> 32, offset mod 2**32, offset >> 32),
        q = i >> 2.
    Because ``i`` is the index in the unsharded tensor, the draw of an element
    does not depend on how many ranks the sequence is split over.
    """
    idx = np.asarray(elem_index, dtype=np.uint64)
    q = idx >> np.uint64(2)
    lane = (idx & np.uint64(3)).astype(np.int64)
    seed = int(seed)
    offset = int(offset)
    ctr = (q & _LO32,
           q >> _SH32,
           np.full(q.shape, offset & 0xFFFFFFFF, dtype=np.uint64),
           np.full(q.shape, (offset >> 32) & 0xFFFFFFFF, dtype=np.uint64))
    words = philox4x32(ctr, (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF))
    stacked = np.stack(words, axis=0)
    return np.take_along_axis(stacked, lane[None, ...], axis=0)[0]
