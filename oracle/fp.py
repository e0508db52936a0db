"""Exact floating-point rounding helpers for the oracle (numpy, no GPU code).

* fp32 operations are numpy float32 operations: IEEE-754 binary32 with
  round-to-nearest-even, which is what the quantizer specification states.
* fp16 conversions: numpy's float32 -> float16 cast rounds to nearest even;
  round-toward-+inf is that cast stepped up by one ulp when it fell below.
* bfloat16: the upper 16 bits of a binary32; rounding to nearest with ties to
  the even upper half, done on the bit pattern (finite inputs; values that
  round past the largest bfloat16 become infinities, as in the format).
* OCP FP8 E4M3 ("e4m3fn"): sign, 4 exponent bits (bias 7), 3 mantissa bits,
  no infinities, 0x7F/0xFF are NaN, largest finite 448, smallest subnormal
  2^-9.  Rounding is to the nearest finite value, ties to the even code, and
  anything beyond 448 in magnitude saturates to +-448.  The value table is
  built from the bit-level definition.
"""
from __future__ import annotations

import numpy as np

FP16_MAX = 65504.0


def f32(x):
    return np.asarray(x, dtype=np.float32)


def fp16_rn(x32) -> np.ndarray:
    """Nearest-even fp16 of float32 values (returned as float16)."""
    return np.asarray(x32, dtype=np.float32).astype(np.float16)


def fp16_ru(x) -> np.ndarray:
    """Smallest fp16 value >= x (x float32 or float64)."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        h = x.astype(np.float16)
    low = h.astype(np.float64) < x
    h = np.where(low, np.nextafter(h, np.float16(np.inf)), h)
    return h.astype(np.float16)


def fp32_ru(x) -> np.ndarray:
    """Smallest float32 value >= x (x float64)."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)
    low = f.astype(np.float64) < x
    return np.where(low, np.nextafter(f, np.float32(np.inf)), f).astype(np.float32)


def bf16_rn(x) -> np.ndarray:
    """Nearest-even bfloat16 of float32 values, returned as float32 (exact)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def _e4m3_table():
    codes = np.arange(256, dtype=np.int64)
    sign = np.where(codes & 0x80, -1.0, 1.0)
    e = (codes >> 3) & 0xF
    m = codes & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0)) * sign
    nan = (codes & 0x7F) == 0x7F
    return val, nan


E4M3_VALUES, E4M3_NAN = _e4m3_table()
E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    out = E4M3_VALUES[codes.astype(np.int64)]
    return np.where(E4M3_NAN[codes.astype(np.int64)], np.nan, out)


# non-negative finite codes 0x00..0x7E in increasing value order
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALS = E4M3_VALUES[_POS_CODES]


def e4m3_rn_satfinite(x) -> np.ndarray:
    """Encode float values to E4M3 codes (uint8): nearest, ties to even code, saturating."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_POS_VALS, a, side="left"), 0, len(_POS_VALS) - 1)
    lo = np.clip(hi - 1, 0, len(_POS_VALS) - 1)
    dlo = a - _POS_VALS[lo]
    dhi = _POS_VALS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo])
    code = np.where(np.signbit(x) & (code != 0), code | 0x80, code)
    code = np.where(np.signbit(x) & (code == 0), 0x80, code)   # keep the sign of -0 / tiny negatives
    return code.astype(np.uint8)
