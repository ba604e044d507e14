"""Counter-based dropout keep mask (oracle side; test infrastructure only).

The WGSL backward page ("flash_attention_v2_backward.wgsl", header comment and
both entry points) multiplies by ``dropout_scale(p, seed, bh, qi, kj)`` whose
hash lives in a file that is not on the pages.  The generator is therefore
fixed by this library's own specification, written from the published
definition of Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
Numbers: As Easy as 1, 2, 3", SC'11, section 4.2):

  * key     = (seed & 0xffffffff, seed >> 32)
  * counter = (qi >> 2, kj, bh, 0) with bh = b * num_heads + h
  * word    = output word (qi & 3) of Philox4x32-10(counter, key)
  * keep    iff word >= T,   T = min(floor(p * 2^32), 2^32 - 1)  (p = 0 keeps all)
  * M_ij    = keep ? 1 / (1 - p) : 0

The bit pattern relative to the pages' own hash is "parity unpinned" (its
source is not published); this implementation is pinned to the published
known-answer vectors of Philox4x32-10 and to keep-rate statistics.
"""
from __future__ import annotations

import numpy as np

# Round multipliers and Weyl key increments of Philox4x32 (SC'11, table 2 and
# section 4.2: the golden ratio and sqrt(3)-1 in 32-bit fixed point).
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
MASK32 = np.uint64(0xFFFFFFFF)


def _mulhilo(a: int, b: np.ndarray):
    prod = np.uint64(a) * b.astype(np.uint64)
    return (prod >> np.uint64(32)) & MASK32, prod & MASK32


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Philox4x32 with 10 rounds on arrays of 32-bit counters.

    One round maps (c0,c1,c2,c3) to
    (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0));
    the key is bumped by the Weyl constants between rounds.
    Returns four uint64 arrays holding 32-bit words.
    """
    c = [np.asarray(x, dtype=np.uint64) & MASK32 for x in (c0, c1, c2, c3)]
    c = list(np.broadcast_arrays(*c))
    ka, kb = int(k0) & 0xFFFFFFFF, int(k1) & 0xFFFFFFFF
    for r in range(10):
        if r > 0:
            ka = (ka + PHILOX_W0) & 0xFFFFFFFF
            kb = (kb + PHILOX_W1) & 0xFFFFFFFF
        hi0, lo0 = _mulhilo(PHILOX_M0, c[0])
        hi1, lo1 = _mulhilo(PHILOX_M1, c[2])
        c = [hi1 ^ c[1] ^ np.uint64(ka), lo1, hi0 ^ c[3] ^ np.uint64(kb), lo0]
    return c


def keep_threshold(p: float) -> int:
    """T = min(floor(p * 2^32), 2^32 - 1), from the fp32 dropout probability."""
    t = int(np.floor(np.float64(np.float32(p)) * 4294967296.0))
    return min(max(t, 0), 0xFFFFFFFF)


def keep_mask(seed: int, bh: int, seq_q: int, seq_k: int, p: float) -> np.ndarray:
    """Boolean keep mask [seq_q, seq_k] of one (batch, head) slice."""
    if p <= 0.0:
        return np.ones((seq_q, seq_k), dtype=bool)
    qi = np.arange(seq_q, dtype=np.uint64)[:, None]
    kj = np.arange(seq_k, dtype=np.uint64)[None, :]
    words = philox4x32_10(qi >> np.uint64(2), kj, np.uint64(bh), np.uint64(0),
                          seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    sel = (qi & np.uint64(3)).astype(np.int64)
    stacked = np.stack(np.broadcast_arrays(*words), axis=0)  # [4, Sq, Sk]
    w = np.take_along_axis(stacked, np.broadcast_to(sel, (seq_q, seq_k))[None], axis=0)[0]
    return w >= np.uint64(keep_threshold(p))


def dropout_multiplier(seed: int, bh: int, seq_q: int, seq_k: int, p: float) -> np.ndarray:
    """M_ij in fp64: 1/(1-p) where kept, 0 where dropped; all ones for p = 0."""
    if p <= 0.0:
        return np.ones((seq_q, seq_k), dtype=np.float64)
    keep = keep_mask(seed, bh, seq_q, seq_k, p)
    return np.where(keep, 1.0 / (1.0 - np.float64(np.float32(p))), 0.0)
