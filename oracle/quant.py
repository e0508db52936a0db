"""Write path of the oracle: the three cache schemes and the band-norm witness.

Every fp32 step is a numpy float32 operation (IEEE round-to-nearest-even), so
codes and scales follow the same sequence of roundings the CUDA writer is
specified to take; reconstructions x_hat, residuals and witnesses are float64.

Band layout.  RoPE in the rotate-half form pairs dim i with dim i+64
(i = 0..63) at frequency base^(-2i/d).  Band b (b = 0..15) is the union of the
four whole pairs i = 4b..4b+3, i.e. dims {4b..4b+3} U {64+4b..64+4b+3}: eight
dims per band, sixteen bands [WitCert summary, Lemma 1: RoPE acts unitarily
within a frequency band; witness of B bands stored at write time].
"""
from __future__ import annotations

import numpy as np

from .fp import FP16_MAX, bf16_rn, e4m3_decode, e4m3_rn_satfinite, fp16_rn, fp16_ru

D = 128
N_BANDS = 16
GROUP = 32
BLOCK = 16

BAND_DIMS = np.array([[4 * b + i for i in range(4)] + [64 + 4 * b + i for i in range(4)]
                      for b in range(N_BANDS)])


# --------------------------------------------------------------------------- witness

def witness(resid: np.ndarray) -> np.ndarray:
    """w_{t,b} = ||r_{t,b}||_2 over each band's eight dims [WitCert summary, witness paragraph]."""
    r = np.asarray(resid, dtype=np.float64)
    return np.sqrt(np.sum(r[..., BAND_DIMS] ** 2, axis=-1))


WITNESS_MARGIN = 2.0 ** -48


def witness_stored(w64: np.ndarray) -> np.ndarray:
    """Stored fp16 witness: smallest fp16 >= w*(1+2^-48).

    Rounding up keeps the stored witness an upper bound of the exact norm, so
    Tier A stays sound after storage; the 2^-48 factor covers the last-bit error
    of a float64 norm.
    """
    return fp16_ru(np.asarray(w64, dtype=np.float64) * (1.0 + WITNESS_MARGIN))


def value_witness(resid: np.ndarray) -> np.ndarray:
    """wv_t = ||r_t||_2 over all 128 dims of a value row's residual r = v - v_hat.

    The value side of the witness idea: the output error the value compression
    adds at the compressed weights is bounded by sum_t p~_t wv_t (triangle
    inequality), with no query involved, so one norm per token suffices.
    """
    r = np.asarray(resid, dtype=np.float64)
    return np.sqrt(np.sum(r ** 2, axis=-1))


# --------------------------------------------------------------------------- INT8 + subtractive dither

def write_int8_dither(x, xi):
    """Subtractively dithered INT8 with per-(token, 32-channel group) scales.

    x_hat = s * (round(x/s + xi) - xi) [WitCert summary, Tier B paragraph], with
        amax = max |x| over the group               (fp32, exact)
        s32  = fp32(amax / 127)                      (fp32 division, nearest)
        s    = min(fp16 round-up(s32), 65504)        (stored scale)
        z    = fp32(fp32(x / s) + xi)                (two fp32 roundings, no FMA)
        code = clamp(rint(z), -128, 127)             (rint: half to even)
    and code = 0 for an all-zero group (s = 0).

    x, xi: float32 [n, 128].  Returns codes int8 [n,128], scales float16 [n,4],
    x_hat float64 [n,128] and the number of clamped codes.
    """
    x = np.asarray(x, dtype=np.float32)
    xi = np.asarray(xi, dtype=np.float32)
    n = x.shape[0]
    g = x.reshape(n, D // GROUP, GROUP)
    xg = xi.reshape(n, D // GROUP, GROUP)
    amax = np.max(np.abs(g), axis=-1)
    s32 = (amax / np.float32(127.0)).astype(np.float32)
    s16 = np.minimum(fp16_ru(s32).astype(np.float32), np.float32(FP16_MAX)).astype(np.float16)
    s = s16.astype(np.float32)[..., None]
    ok = s > 0
    v = (g / np.where(ok, s, np.float32(1.0))).astype(np.float32)
    z = (v + xg).astype(np.float32)
    r = np.rint(z)
    clamps = int(np.sum(ok & ((r < -128) | (r > 127))))
    code = np.where(ok, np.clip(r, -128, 127), 0).astype(np.int8)
    xhat = s.astype(np.float64) * (code.astype(np.float64) - xg.astype(np.float64))
    return code.reshape(n, D), s16, xhat.reshape(n, D), clamps


# --------------------------------------------------------------------------- raw-cast FP8

def write_fp8(x):
    """Black-box raw cast to OCP E4M3 (nearest-even, saturating), no scale
    [WitCert summary, gate results: raw-cast fp8].  Returns codes uint8 and x_hat."""
    code = e4m3_rn_satfinite(np.asarray(x, dtype=np.float32))
    return code, e4m3_decode(code)


# --------------------------------------------------------------------------- black-box tensor function

def write_blackbox(x_hat):
    """Any scheme given as one tensor function f [WitCert abstract: any scheme
    registered as one tensor function is measured; Tier A is sound for any
    cache-preserving black-box quantizer].  The caller applies f; the cache keeps
    its output as bfloat16 (nearest even of the float32 value), and the decode and
    the witness both use that stored value.  x_hat: float32 [n, 128]."""
    return bf16_rn(np.asarray(x_hat, dtype=np.float32)).astype(np.float64)


# --------------------------------------------------------------------------- KIVI-style 2-bit

def _asym2(x, axis):
    """Asymmetric 2-bit quantization along `axis` (min/max, 4 levels).

        d32   = fp32(max - min)
        scale = fp16 nearest(fp32(d32 / 3))    zero = fp16 nearest(min)   (both clamped to +-65504)
        code  = clamp(rint(fp32(fp32(x - zero) / scale)), 0, 3)   (0 when scale = 0)
        x_hat = zero + scale * code
    """
    x = np.asarray(x, dtype=np.float32)
    mn = np.min(x, axis=axis, keepdims=True)
    mx = np.max(x, axis=axis, keepdims=True)
    d32 = (mx - mn).astype(np.float32)
    s32 = (d32 / np.float32(3.0)).astype(np.float32)
    lim = np.float32(FP16_MAX)
    scale = fp16_rn(np.clip(s32, -lim, lim))
    zero = fp16_rn(np.clip(mn, -lim, lim))
    sc = scale.astype(np.float32)
    zr = zero.astype(np.float32)
    ok = sc > 0
    num = (x - zr).astype(np.float32)
    v = (num / np.where(ok, sc, np.float32(1.0))).astype(np.float32)
    code = np.where(ok, np.clip(np.rint(v), 0, 3), 0).astype(np.uint8)
    xhat = zr.astype(np.float64) + sc.astype(np.float64) * code.astype(np.float64)
    return code, scale, zero, xhat


def write_kivi2_k(block):
    """KIVI keys: per channel over one full 16-token block.  block: float32 [16, 128].
    Returns codes [16,128], scale [128], zero [128], x_hat [16,128]."""
    code, scale, zero, xhat = _asym2(block, axis=0)
    return code, scale[0], zero[0], xhat


def write_kivi2_v(x):
    """KIVI values: per token over each 32-channel group.  x: float32 [n, 128].
    Returns codes [n,128], scale [n,4], zero [n,4], x_hat [n,128]."""
    n = x.shape[0]
    code, scale, zero, xhat = _asym2(np.asarray(x, np.float32).reshape(n, D // GROUP, GROUP), axis=-1)
    return code.reshape(n, D), scale[..., 0], zero[..., 0], xhat.reshape(n, D)


# --------------------------------------------------------------------------- byte accounting

BYTES_PER_TOKEN_HEAD = {
    # K codes + V codes + K scales + V scales + K witness
    "int8_dither": 128 + 128 + 8 + 8 + 32,
    "int8_rtn": 128 + 128 + 8 + 8 + 32,
    # K codes + V codes + K witness
    "fp8_e4m3": 128 + 128 + 32,
    # K codes + K (scale, zero) per channel per 16 tokens + V codes + V (scale, zero) per group + K witness
    "kivi2": 32 + (128 * 2 * 2) // BLOCK + 32 + 4 * 2 * 2 + 32,
    # K_hat + V_hat as bfloat16 + K witness
    "blackbox": 256 + 256 + 32,
}
# optional value witness: one fp16 norm per token and head
V_WITNESS_BYTES = 2
