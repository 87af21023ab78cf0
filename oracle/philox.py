"""Philox4x32-10 counter-based generator.  TEST INFRASTRUCTURE ONLY.

Written from the definition in Salmon, Moraes, Dror, Shaw, "Parallel Random
Numbers: As Easy as 1, 2, 3" (SC'11), §4.2 (Philox) and Table 2 (round
constants).  A Philox4x32 round maps the counter (c0, c1, c2, c3) under the
round key (k0, k1) to

    (hi(M1·c2) ^ c1 ^ k0,  lo(M1·c2),  hi(M0·c0) ^ c3 ^ k1,  lo(M0·c0))

with 32x32->64-bit products split into high and low words, and the key is
bumped by the Weyl constants (W0, W1) between rounds; ten rounds are applied.

The method draws its randomness from a generator keyed by the layer step's
seed (stochastic rounding on gradients and the random sign vector of the
Hadamard transform: Pretraining Large Language Models with NVFP4, Resumo
técnico §2, items 2 and 4).  The pages do not name a generator; Philox is the
counter-based choice so that every element's bits are a pure function of
(seed, stream, index).
"""

import numpy as np

PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint32(0x9E3779B9)
PHILOX_W1 = np.uint32(0xBB67AE85)
_MASK32 = np.uint64(0xFFFFFFFF)


def _mulhilo(a_u64, b_u32_as_u64):
    p = a_u64 * b_u32_as_u64  # < 2^64, no overflow
    return (p >> np.uint64(32)).astype(np.uint32), (p & _MASK32).astype(np.uint32)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Ten Philox4x32 rounds.  Counters are broadcastable uint32 arrays; the key
    is two uint32 scalars.  Returns four uint32 arrays."""
    c = [np.asarray(x, dtype=np.uint32) for x in (c0, c1, c2, c3)]
    c = np.broadcast_arrays(*c)
    c = [x.astype(np.uint32).copy() for x in c]
    k0 = np.uint32(k0)
    k1 = np.uint32(k1)
    for rnd in range(10):
        if rnd > 0:
            k0 = np.uint32((int(k0) + int(PHILOX_W0)) & 0xFFFFFFFF)
            k1 = np.uint32((int(k1) + int(PHILOX_W1)) & 0xFFFFFFFF)
        hi0, lo0 = _mulhilo(PHILOX_M0, c[0].astype(np.uint64))
        hi1, lo1 = _mulhilo(PHILOX_M1, c[2].astype(np.uint64))
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return c


def seed_key(seed):
    """64-bit seed -> Philox key (low word, high word)."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return seed & 0xFFFFFFFF, seed >> 32


def sr_uniform16(seed, stream_id, elem_index):
    """The 16-bit uniform used to stochastically round element ``elem_index``.

    Element e takes Philox(key = seed, counter = (lo32(e // 8), hi32(e // 8),
    stream_id, 0)); of the four output words it uses word (e mod 8) // 2, its
    low half for even e and its high half for odd e.  One Philox call serves
    eight consecutive elements of the quantized tensor's row-major order.
    """
    e = np.asarray(elem_index, dtype=np.uint64)
    g = e >> np.uint64(3)
    k0, k1 = seed_key(seed)
    w = philox4x32_10((g & _MASK32).astype(np.uint32), (g >> np.uint64(32)).astype(np.uint32),
                      np.uint32(stream_id), np.uint32(0), k0, k1)
    words = np.stack(w, axis=0)
    sel = ((e & np.uint64(7)) >> np.uint64(1)).astype(np.int64)
    word = np.take_along_axis(words.reshape(4, -1), sel.reshape(1, -1), axis=0).reshape(e.shape)
    half = (e & np.uint64(1)).astype(np.uint32)
    return np.where(half == 0, word & np.uint32(0xFFFF), word >> np.uint32(16)).astype(np.uint32)
