"""Philox4x32-10 counter-based generator (Salmon, Moraes, Dror, Shaw,
"Parallel random numbers: as easy as 1, 2, 3", SC'11), written from the
published definition and vectorised with numpy.

The uniforms that speculative-sampling verification consumes are drawn here
once and handed, unchanged, to both the CUDA path and the oracle.  Nothing in
this file is part of the verification arithmetic.

Definition used:
  round(c, k):  (hi0, lo0) = mulhilo(0xD2511F53, c0)
                (hi1, lo1) = mulhilo(0xCD9E8D57, c2)
                c' = (hi1 ^ c1 ^ k0,  lo1,  hi0 ^ c3 ^ k1,  lo0)
  key bump:     k0 += 0x9E3779B9,  k1 += 0xBB67AE85   (mod 2^32)
  Philox4x32-10: ten rounds, the key bumped between consecutive rounds.
"""
from __future__ import annotations

import numpy as np

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK = np.uint64(0xFFFFFFFF)
_SH = np.uint64(32)


def philox4x32_10(counter, key):
    """Apply Philox4x32-10.

    counter: uint array of shape [..., 4] (32-bit words c0..c3).
    key:     uint array of shape [..., 2] or a pair (k0, k1), broadcastable.
    Returns a uint32 array of shape [..., 4].
    """
    c = np.asarray(counter, dtype=np.uint64) & _MASK
    k = np.asarray(key, dtype=np.uint64) & _MASK
    c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
    k0 = np.broadcast_to(k[..., 0], c0.shape).copy()
    k1 = np.broadcast_to(k[..., 1], c0.shape).copy()
    for r in range(10):
        if r:
            k0 = (k0 + np.uint64(_W0)) & _MASK
            k1 = (k1 + np.uint64(_W1)) & _MASK
        p0 = _M0 * c0
        p1 = _M1 * c2
        hi0, lo0 = p0 >> _SH, p0 & _MASK
        hi1, lo1 = p1 >> _SH, p1 & _MASK
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def philox_uniforms(n: int, seed: int = 0, offset: int = 0) -> np.ndarray:
    """n float32 uniforms in [0, 1).

    Element j uses counter (offset + j, 0, 0, 0) and key (seed, 0); the value
    is the top 24 bits of output word 0 times 2^-24, which is exact in both
    float32 and float64.
    """
    idx = np.arange(offset, offset + n, dtype=np.uint64)
    ctr = np.zeros((n, 4), dtype=np.uint64)
    ctr[:, 0] = idx & _MASK
    ctr[:, 1] = idx >> _SH
    out = philox4x32_10(ctr, np.array([seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF], dtype=np.uint64))
    x0 = out[:, 0].astype(np.uint32)
    return ((x0 >> np.uint32(8)).astype(np.float64) * 2.0 ** -24).astype(np.float32)
