"""Philox4x32-10 and the dither stream, written from the published definition.

Philox is the counter-based generator of Salmon, Moraes, Dror and Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11): ten rounds, each of
which multiplies counter words 0 and 2 by two fixed odd constants, splits the
64-bit products into high and low halves, and recombines them with the other
two counter words and the round key; the key is advanced by two Weyl
increments between rounds.

The dither stream is this module's reading of the Tier B paragraph's
requirement that the decoder recompute the writer's dither exactly rather than
store it [WitCert summary, Tier B paragraph]; it is keyed on (layer, head,
token, channel):

    key     = (seed mod 2^32, seed div 2^32)
    counter = (token position t, (channel // 4) | (tensor << 16),
               kv_head | (layer << 16), 0)              tensor: 0 = K, 1 = V
    u       = output word (channel mod 4)
    xi      = (u >> 8) * 2^-24 - 1/2                    exact in fp32, in [-1/2, 1/2)

There is no sequence id in the counter, so every sequence sees the same dither
at the same (layer, head, position, channel).
"""
from __future__ import annotations

import numpy as np

MASK32 = np.uint64(0xFFFFFFFF)
_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = np.uint64(0x9E3779B9)
_W1 = np.uint64(0xBB67AE85)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Ten Philox rounds on broadcastable arrays of 32-bit words (held as uint64)."""
    c0, c1, c2, c3, k0, k1 = (np.asarray(a, dtype=np.uint64) & MASK32 for a in (c0, c1, c2, c3, k0, k1))
    c0, c1, c2, c3 = np.broadcast_arrays(c0, c1, c2, c3)
    for r in range(10):
        if r:
            k0 = (k0 + _W0) & MASK32
            k1 = (k1 + _W1) & MASK32
        p0 = _M0 * c0            # < 2^64: exact in uint64
        p1 = _M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & MASK32, lo1, (hi0 ^ c3 ^ k1) & MASK32, lo0
    return c0, c1, c2, c3


def dither(seed: int, layer: int, kv_head: int, positions, tensor: int, d: int = 128) -> np.ndarray:
    """Dither xi for the given token positions: float32 array [len(positions), d]."""
    t = np.asarray(positions, dtype=np.uint64).reshape(-1, 1)
    quad = np.arange(d // 4, dtype=np.uint64).reshape(1, -1)
    k0 = np.uint64(seed & 0xFFFFFFFF)
    k1 = np.uint64((seed >> 32) & 0xFFFFFFFF)
    w1 = quad | np.uint64(tensor << 16)
    w2 = np.uint64(kv_head | (layer << 16))
    out = philox4x32_10(t, w1, w2, np.uint64(0), k0, k1)        # four [n, d/4] arrays
    u = np.stack(out, axis=-1).reshape(t.shape[0], d)           # channel c <- word c % 4
    xi = (u >> np.uint64(8)).astype(np.float64) * 2.0 ** -24 - 0.5
    return xi.astype(np.float32)                                 # exact conversion
