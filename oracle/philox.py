"""Philox4x32-10 counter-based generator, oracle side (numpy, vectorised).

TEST INFRASTRUCTURE: imported only by tests/, __graft_entry__.smoke() and
bench.py's CPU-baseline leg. The CUDA path carries its own implementation and
shares nothing with this file.

Written from the published definition in Salmon, Moraes, Dror and Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), section 4: a 4-word
counter and a 2-word key; each of the 10 rounds multiplies counter words 0 and
2 by two fixed odd constants, swaps the halves of the 64-bit products into
the counter while XOR-ing in the other two counter words and the round key,
and the key is advanced by two Weyl increments between rounds.

Stream layout used by the sampler's exponential race (one word per token):
    key     = (seed mod 2^32, seed >> 32)
    counter = (token id, row, step mod 2^32, step >> 32)
    u       = (2 * (word0 >> 9) + 1) * 2^-24    in (0, 1), exact in f32 and f64
The race draws for a token therefore do not depend on which other tokens are
candidates, so a subset pass and a full pass draw the same token (the Gaudi
"topk-subset-sampler" page, section "The fix", notes that its subset path
does not have this property).
"""
from __future__ import annotations

import numpy as np

_MUL0 = np.uint64(0xD2511F53)
_MUL1 = np.uint64(0xCD9E8D57)
_WEYL0 = np.uint64(0x9E3779B9)
_WEYL1 = np.uint64(0xBB67AE85)
_LO32 = np.uint64(0xFFFFFFFF)
_SH32 = np.uint64(32)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Return the four 32-bit output words for counters (c0..c3) under key (k0, k1).

    All arguments broadcast; results are uint32 arrays.
    """
    x0 = np.asarray(c0, dtype=np.uint64) & _LO32
    x1 = np.asarray(c1, dtype=np.uint64) & _LO32
    x2 = np.asarray(c2, dtype=np.uint64) & _LO32
    x3 = np.asarray(c3, dtype=np.uint64) & _LO32
    y0 = np.asarray(k0, dtype=np.uint64) & _LO32
    y1 = np.asarray(k1, dtype=np.uint64) & _LO32
    for _ in range(10):
        p0 = _MUL0 * x0  # < 2^64: both factors are below 2^32
        p1 = _MUL1 * x2
        x0, x1, x2, x3 = ((p1 >> _SH32) ^ x1 ^ y0) & _LO32, p1 & _LO32, ((p0 >> _SH32) ^ x3 ^ y1) & _LO32, p0 & _LO32
        y0 = (y0 + _WEYL0) & _LO32
        y1 = (y1 + _WEYL1) & _LO32
    return (x0.astype(np.uint32), x1.astype(np.uint32), x2.astype(np.uint32), x3.astype(np.uint32))


def race_uniform(seed: int, step: int, row: int, token_ids) -> np.ndarray:
    """Uniform variates in (0, 1) for the given tokens of one row at one decode step (float64)."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    step = int(step) & 0xFFFFFFFFFFFFFFFF
    ids = np.asarray(token_ids, dtype=np.uint64)
    w0, _, _, _ = philox4x32_10(ids, np.uint64(row), np.uint64(step & 0xFFFFFFFF), np.uint64(step >> 32),
                                np.uint64(seed & 0xFFFFFFFF), np.uint64(seed >> 32))
    return (2.0 * (w0 >> np.uint32(9)).astype(np.float64) + 1.0) * 2.0 ** -24
