"""Pins of the oracle's write path: Philox, dither, the three schemes, the witness.

Each check compares the oracle with something other than its own formula:
published test vectors, format definitions, closed forms, a library cast,
brute force over every code, or a statistical law the pages cite.
"""
import math
import os

import numpy as np
import pytest
import scipy.stats as st
import torch

from oracle import fp, quant
from oracle.philox import dither, philox4x32_10
from workload import bf16_round

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------- Philox

def test_philox_known_answer_vectors():
    """Random123's published Philox4x32-10 vectors (tests/golden/philox4x32_10_kat.txt)."""
    n = 0
    for line in open(os.path.join(GOLD, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(x, 16) for x in line.split()]
        out = philox4x32_10(*w[:6])
        assert [int(o) for o in out] == w[6:]
        n += 1
    assert n == 3


def test_dither_grid_range_and_uniformity():
    xi = dither(0, 3, 1, np.arange(4096), 0).astype(np.float64)
    assert xi.min() >= -0.5 and xi.max() < 0.5
    # exact multiples of 2^-24 (24-bit fixed point)
    assert np.all(np.floor(xi * 2 ** 24) == xi * 2 ** 24)
    ks = st.kstest(xi.ravel() + 0.5, "uniform")
    assert ks.pvalue > 1e-3
    # distinct streams for K/V, heads, layers, seeds; reproducible
    assert not np.array_equal(xi, dither(0, 3, 1, np.arange(4096), 1))
    assert not np.array_equal(xi, dither(0, 3, 2, np.arange(4096), 0))
    assert not np.array_equal(xi, dither(0, 4, 1, np.arange(4096), 0))
    assert not np.array_equal(xi, dither(1, 3, 1, np.arange(4096), 0))
    np.testing.assert_array_equal(dither(0, 3, 1, [17, 900], 0), xi[[17, 900]])


def test_dither_channel_independence():
    xi = dither(7, 0, 0, np.arange(20000), 1).astype(np.float64)
    c = np.corrcoef(xi[:, :8].T)
    off = c[~np.eye(8, dtype=bool)]
    assert np.max(np.abs(off)) < 0.05


# --------------------------------------------------------------------------- INT8 dither

def _rand_x(rng, n, scale_outliers=True):
    x = rng.standard_normal((n, 128)).astype(np.float32)
    if scale_outliers:
        x[:, [10, 74]] *= 50
    return bf16_round(x)


def test_int8_codes_are_nearest_levels_by_brute_force():
    """code = the nearest integer to fp32(fp32(x/s)+xi), ties to even, found by scanning all 256 codes."""
    rng = np.random.default_rng(1)
    x = _rand_x(rng, 64)
    xi = dither(0, 0, 0, np.arange(64), 0)
    code, s16, xhat, clamps = quant.write_int8_dither(x, xi)
    assert clamps == 0
    s = s16.astype(np.float32)
    z = ((x.reshape(64, 4, 32) / s[..., None]).astype(np.float32) + xi.reshape(64, 4, 32)).astype(np.float32)
    z = z.reshape(64, 128).astype(np.float64)
    levels = np.arange(-128, 128, dtype=np.float64)
    dist = np.abs(z[..., None] - levels)
    nearest = dist == dist.min(-1, keepdims=True)
    # among equally near levels take the even one
    score = np.where(nearest, (levels % 2 != 0).astype(np.float64), np.inf)
    pick = levels[np.argmin(score, -1)]
    np.testing.assert_array_equal(code.astype(np.float64), pick)
    # the scale bounds the group's amax
    amax = np.abs(x.reshape(64, 4, 32)).max(-1)
    assert np.all(s.astype(np.float64) * 127 >= amax * (1 - 2 ** -23))


def test_int8_round_half_even_and_zero_group():
    x = np.zeros((1, 128), np.float32)
    x[0, :32] = 127.0                       # amax 127 -> s = 1
    x[0, 1], x[0, 2], x[0, 3] = 2.5, 3.5, -2.5
    xi = np.zeros((1, 128), np.float32)
    code, s16, xhat, _ = quant.write_int8_dither(x, xi)
    assert float(s16[0, 0]) == 1.0
    assert (code[0, 1], code[0, 2], code[0, 3]) == (2, 4, -2)
    assert np.all(code[0, 32:] == 0) and np.all(s16[0, 1:] == 0)
    assert np.all(xhat[0, 32:] == 0)


def test_int8_dither_residual_is_uniform_and_input_independent():
    """Subtractive dither: r = x - x_hat is U[-s/2, s/2) whatever x is (classical dither theory,
    [WitCert summary, Tier B paragraph])."""
    rng = np.random.default_rng(2)
    n = 50000
    base = np.linspace(-1.0, 1.0, 32, dtype=np.float32)
    x = np.tile(np.concatenate([base * 127 / 1.0] * 4), (n, 1)).astype(np.float32)
    x[:, 5] = 0.3                          # fixed input values inside group 0
    x[:, 6] = 0.8
    xi = (rng.integers(0, 2 ** 24, size=(n, 128)) * 2.0 ** -24 - 0.5).astype(np.float32)
    code, s16, xhat, _ = quant.write_int8_dither(x, xi)
    s = float(s16[0, 0])
    for c in (5, 6, 17):
        r = (x[:, c] - xhat[:, c]) / s
        assert r.min() >= -0.5 - 1e-6 and r.max() <= 0.5 + 1e-6
        assert st.kstest(r + 0.5, "uniform").pvalue > 1e-3
        assert abs(r.mean()) < 4 * math.sqrt(1 / 12 / n)
        assert abs(r.var() - 1 / 12) < 0.003
    # independence from the input: random inputs, correlation ~ 0
    xr = _rand_x(rng, n, scale_outliers=False)
    _, s16r, xhr, _ = quant.write_int8_dither(xr, xi)
    rr = (xr - xhr) / np.repeat(s16r.astype(np.float64), 32, axis=1)
    assert abs(np.corrcoef(rr[:, 3], xr[:, 3])[0, 1]) < 0.02


# --------------------------------------------------------------------------- FP8 E4M3

def test_e4m3_format_points():
    for line in open(os.path.join(GOLD, "e4m3_points.txt")):
        if line.startswith("#") or not line.strip():
            continue
        v, c = line.split()
        got = int(fp.e4m3_rn_satfinite(np.array([float(v)]))[0])
        assert got == int(c, 16), (v, hex(got))
    assert fp.E4M3_VALUES[0x7E] == 448.0 and np.isnan(fp.e4m3_decode(np.array([0x7F]))[0])


def test_e4m3_matches_torch_cast_in_range():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.1, 1, 30, 150)]).astype(np.float32)
    x = x[np.abs(x) < 440]
    ours = fp.e4m3_rn_satfinite(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_fp8_write_residual_is_relative():
    rng = np.random.default_rng(4)
    x = _rand_x(rng, 256)
    code, xhat = quant.write_fp8(x)
    rel = np.abs(x - xhat) / np.maximum(np.abs(x), 2 ** -6)
    assert rel.max() <= 2 ** -4 + 1e-12     # half a 3-bit mantissa step


# --------------------------------------------------------------------------- KIVI 2-bit

def test_kivi_levels_and_extremes():
    rng = np.random.default_rng(5)
    blk = _rand_x(rng, 16)
    code, scale, zero, xhat = quant.write_kivi2_k(blk)
    assert code.max() <= 3
    sc = scale.astype(np.float64)
    zr = zero.astype(np.float64)
    lv = zr[None, :] + sc[None, :] * np.arange(4)[:, None]          # [4, 128] the four levels
    # every code is a nearest level (up to fp32 rounding at exact midpoints)
    dist = np.abs(blk[:, None, :].astype(np.float64) - lv[None])   # [16, 4, 128]
    chosen = np.take_along_axis(dist, code[:, None, :].astype(np.int64), 1)[:, 0]
    assert np.all(chosen <= dist.min(1) + 1e-6 * np.abs(blk).max())
    # the channel minimum maps to level 0, the maximum to level 3
    assert np.all(code[np.argmin(blk, 0), np.arange(128)] == 0)
    assert np.all(code[np.argmax(blk, 0), np.arange(128)] == 3)
    # a constant channel reconstructs exactly
    blk2 = blk.copy()
    blk2[:, 7] = np.float32(0.75)
    c2, _, _, xh2 = quant.write_kivi2_k(blk2)
    assert np.all(c2[:, 7] == 0) and np.all(xh2[:, 7] == 0.75)


def test_kivi_v_per_token_groups():
    rng = np.random.default_rng(6)
    v = _rand_x(rng, 10, scale_outliers=False)
    code, scale, zero, xhat = quant.write_kivi2_v(v)
    assert scale.shape == (10, 4)
    step = np.repeat(scale.astype(np.float64), 32, axis=1)
    assert np.all(np.abs(v - xhat) <= step * 0.5 + 1e-3 * np.abs(v).max() + step * 2 ** -10 * 3)


# --------------------------------------------------------------------------- witness, Lemma 1, Theorem 2

def _rope_rotate(r, pos, base):
    """Rotate-half RoPE of a residual vector at position pos (written out here, not imported)."""
    i = np.arange(64)
    th = pos * base ** (-2.0 * i / 128)
    c, s = np.cos(th), np.sin(th)
    a, b = r[..., :64], r[..., 64:]
    return np.concatenate([a * c - b * s, a * s + b * c], -1)


@pytest.mark.parametrize("base", [1e4, 1e6, 5e6])
def test_lemma1_band_norms_invariant_under_rope(base):
    rng = np.random.default_rng(7)
    r = rng.standard_normal((50, 128))
    w0 = quant.witness(r)
    for pos in (1, 37, 4095, 131071):
        w1 = quant.witness(_rope_rotate(r, pos, base))
        np.testing.assert_allclose(w1, w0, rtol=1e-12, atol=0)
    # negative control: bands of 8 contiguous dims split rotation pairs and are not invariant
    contig = lambda x: np.sqrt((x.reshape(50, 16, 8) ** 2).sum(-1))
    assert np.max(np.abs(contig(_rope_rotate(r, 37, base)) - contig(r))) > 1e-3


def test_witness_stored_rounds_up_within_one_fp16_ulp():
    rng = np.random.default_rng(8)
    w = np.abs(rng.standard_normal(100000)) * np.exp(rng.uniform(-8, 5, 100000))
    ws = quant.witness_stored(w).astype(np.float64)
    assert np.all(ws >= w)
    # one fp16 ulp: 2^-10 relative for normals, 2^-24 absolute below 2^-14 (subnormals)
    assert np.all(ws <= np.maximum(w * (1 + 2 ** -10), w + 2 ** -24) * (1 + 2 ** -40))


@pytest.mark.parametrize("scheme", ["int8_dither", "fp8_e4m3", "kivi2"])
def test_theorem2_cauchy_schwarz_brute_force(scheme):
    """|q.k - q.k_hat|/sqrt(d) <= (1/sqrt d) sum_b ||q_b|| w_b for every token and query
    [WitCert summary, Theorem 2], with the exact and with the stored witness."""
    from oracle import meter
    rng = np.random.default_rng(9)
    k = _rand_x(rng, 256)
    if scheme == "int8_dither":
        _, _, kh, _ = quant.write_int8_dither(k, dither(0, 0, 0, np.arange(256), 0))
    elif scheme == "fp8_e4m3":
        _, kh = quant.write_fp8(k)
    else:
        kh = np.concatenate([quant.write_kivi2_k(k[i:i + 16])[3] for i in range(0, 256, 16)])
    w = quant.witness(k - kh)
    q = rng.standard_normal((64, 128)) * rng.uniform(0.1, 10, (64, 1))
    err = np.abs(q @ (k - kh).T) / math.sqrt(128)
    assert np.all(err <= meter.tier_a(q, w) * (1 + 1e-12))
    assert np.all(err <= meter.tier_a(q, quant.witness_stored(w).astype(np.float64)))


def test_theorem2_is_tight_for_band_aligned_residuals():
    """Equality holds when each band of the residual is parallel to that band of q."""
    from oracle import meter
    rng = np.random.default_rng(10)
    q = rng.standard_normal(128)
    r = np.zeros(128)
    for b in range(16):
        dims = quant.BAND_DIMS[b]
        r[dims] = q[dims] * rng.uniform(0.1, 2.0)
    lhs = abs(q @ r) / math.sqrt(128)
    rhs = meter.tier_a(q[None], quant.witness(r)[None])[0, 0]
    assert abs(lhs - rhs) <= 1e-12 * rhs


def test_bytes_per_token_head():
    assert quant.BYTES_PER_TOKEN_HEAD == {"int8_dither": 304, "fp8_e4m3": 288, "kivi2": 144, "int8_rtn": 304,
                                          "blackbox": 544}
    assert quant.V_WITNESS_BYTES == 2


def test_rtn_writer_is_the_nearest_code_and_idempotent():
    """INT8 round to nearest (the dithered writer with xi = 0): every code is the nearest of the
    256 codes under its group's scale (brute force), and requantizing x_hat returns the same
    codes and values."""
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((6, 128)) * rng.uniform(0.01, 30, (6, 1))).astype(np.float32)
    x[:, 10] *= 50
    c, s, xh, _ = quant.write_int8_dither(x, np.zeros_like(x))
    sg = np.repeat(s.astype(np.float64), 32, axis=1)
    allc = np.arange(-128, 128, dtype=np.float64)
    dist = np.abs(x.astype(np.float64)[..., None] - sg[..., None] * allc)      # [6, 128, 256]
    best = dist.min(-1)
    mine = np.abs(x.astype(np.float64) - sg * c)
    assert np.all(mine <= best * (1 + 1e-12) + 1e-300)
    c2, s2, xh2, _ = quant.write_int8_dither(xh.astype(np.float32), np.zeros_like(x))
    assert np.array_equal(s2, s) and np.array_equal(c2, c) and np.array_equal(xh2, xh)
