"""Pins of the black-box scheme and of the value witness / value meter.

The black-box scheme stores a caller's tensor-function output as bfloat16
[WitCert abstract: any scheme registered as one tensor function is measured;
Tier A holds for any cache-preserving black-box quantizer].  Its pins: the
bfloat16 rounding against torch's cast and hand-worked ties; Theorem 2
(|q.k - q.k^|/sqrt d <= eps_t) and TV <= meter by brute force for arbitrary
tensor functions; the identity function giving zero witness, zero meter and
plain attention.

The value meter E_V = sum_t p~_t wv_t (a reading of this library: the pages define
no value bound) is pinned by the triangle inequality it rests on, checked by
brute force on every scheme, by a residual shared by all tokens (where the
inequality is an equality) and by uniform weights (q = 0: E_V is the mean).
"""
import math

import numpy as np
import torch

from oracle import OracleCache, fp, meter


# --------------------------------------------------------------------------- bfloat16 rounding

def test_bf16_rn_matches_torch_cast():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.uniform(-30, 30, 20000),
                        np.array([0.0, -0.0, 1e-40, -3e-39, 3.3e38, -3.3e38])]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    got = fp.bf16_rn(x)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_bf16_rn_ties_go_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 (odd last bit): to 1.  1 + 3*2^-8 lies
    # halfway between 1 + 2^-7 and 1 + 2^-6 (even): to 1 + 2^-6.  One unit of fp32 past the tie
    # goes up.
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -23, -(1 + 2.0 ** -8)], np.float32)
    assert fp.bf16_rn(x).tolist() == [1.0, 1 + 2.0 ** -6, 1 + 2.0 ** -7, -1.0]


# --------------------------------------------------------------------------- black-box scheme

def _tensor_functions(rng):
    """A few tensor functions of the kind a caller registers: a coarse uniform grid, a
    per-row relative perturbation, a 4-bit-mantissa truncation and sparse large errors."""
    def grid(x):
        return np.round(x * 4.0) / 4.0

    def noisy(x):
        return x * (1.0 + 0.05 * rng.standard_normal(x.shape))

    def trunc4(x):
        m, e = np.frexp(x)
        return np.ldexp(np.trunc(m * 16.0) / 16.0, e)

    def sparse(x):
        y = x.copy()
        mask = rng.random(x.shape) < 0.02
        y[mask] += 3.0 * rng.standard_normal(mask.sum())
        return y
    return [grid, noisy, trunc4, sparse]


def test_blackbox_theorem2_and_tv_bound_by_brute_force():
    """Every token of every tensor function: |q.k - q.k^|/sqrt d <= eps_t (from the stored fp16
    witness), and TV(p, p~) <= the Tier A meter."""
    rng = np.random.default_rng(5)
    S, Hkv, Hq = 96, 2, 4
    K = fp.bf16_rn(rng.standard_normal((1, S, Hkv, 128)).astype(np.float32))
    V = fp.bf16_rn(rng.standard_normal((1, S, Hkv, 128)).astype(np.float32))
    q = rng.standard_normal((1, Hq, 128)) * 3.0
    for f in _tensor_functions(rng):
        c = OracleCache(1, Hq, Hkv, 1, "blackbox")
        c.write(0, K, V, f(K.astype(np.float64)), f(V.astype(np.float64)))
        r = c.decode(0, q, 1e-2)
        for h in range(Hkv):
            kh, vh, w, _, _ = c.group_view(0, 0, h)
            qs = q[0, 2 * h:2 * h + 2]
            exact = qs @ K[0, :, h].astype(np.float64).T / math.sqrt(128)
            comp = qs @ kh.T / math.sqrt(128)
            eps = meter.tier_a(qs, w)
            assert np.all(np.abs(exact - comp) <= eps * (1 + 1e-12) + 1e-12)
            tv = meter.tv_exact(meter.softmax(exact), meter.softmax(comp))
            assert np.all(tv <= r["meter_a"][0, 2 * h:2 * h + 2] * (1 + 1e-12) + 1e-15)
        assert np.all(np.isnan(r["meter_b"]))


def test_blackbox_identity_is_exact_attention():
    rng = np.random.default_rng(6)
    S, Hkv, Hq = 40, 2, 8
    K = fp.bf16_rn(rng.standard_normal((2, S, Hkv, 128)).astype(np.float32))
    V = fp.bf16_rn(rng.standard_normal((2, S, Hkv, 128)).astype(np.float32))
    q = rng.standard_normal((2, Hq, 128))
    c = OracleCache(1, Hq, Hkv, 2, "blackbox", v_witness=True)
    c.write(0, K, V, K, V)
    r = c.decode(0, q, 1e-2)
    assert np.all(c.w16[0] == 0) and np.all(c.wv16[0] == 0)
    assert np.all(r["meter_a"] == 0) and np.all(r["meter_v"] == 0)
    for i in range(2):
        for j in range(Hq):
            _, _, out = meter.attention(q[i, j:j + 1], K[i, :, j // 4], V[i, :, j // 4])
            np.testing.assert_allclose(r["out"][i, j], out[0], rtol=1e-12, atol=1e-12)


def test_blackbox_store_is_the_bf16_of_the_function_output():
    """Stored keys are bf16(f(x)) (fp32 first), so for an output already in bfloat16 the store is
    that output unchanged, and the witness is the band norm of x - f(x) (fp8 cast: every E4M3
    value is a bfloat16, so the black-box store reproduces the FP8 scheme's store)."""
    rng = np.random.default_rng(8)
    K = fp.bf16_rn(rng.standard_normal((1, 32, 1, 128)).astype(np.float32) * 4)
    V = fp.bf16_rn(rng.standard_normal((1, 32, 1, 128)).astype(np.float32))
    f = lambda x: fp.e4m3_decode(fp.e4m3_rn_satfinite(x))
    bb = OracleCache(1, 2, 1, 1, "blackbox")
    bb.write(0, K, V, f(K), f(V))
    f8 = OracleCache(1, 2, 1, 1, "fp8_e4m3")
    f8.write(0, K, V)
    assert np.array_equal(bb.khat[0], f8.khat[0]) and np.array_equal(bb.vhat[0], f8.vhat[0])
    assert np.array_equal(bb.w16[0], f8.w16[0])
    # a non-bf16 output is rounded to nearest even bfloat16 before anything uses it
    x = np.full((1, 1, 1, 128), 1 + 2.0 ** -8 + 2.0 ** -20, np.float32)
    c = OracleCache(1, 2, 1, 1, "blackbox")
    c.write(0, np.ones_like(x), np.ones_like(x), x, x)
    assert np.all(c.khat[0] == 1 + 2.0 ** -7)


# --------------------------------------------------------------------------- value witness / meter

def test_value_meter_bounds_the_value_error_on_every_scheme():
    """|| sum_t p~_t v_t - sum_t p~_t v^_t || <= E_V for every (sequence, query head)."""
    rng = np.random.default_rng(9)
    S, Hkv, Hq, B = 70, 2, 4, 2
    K = fp.bf16_rn(rng.standard_normal((B, S, Hkv, 128)).astype(np.float32))
    V = fp.bf16_rn((rng.standard_normal((B, S, Hkv, 128)) * rng.uniform(0.1, 5, (B, S, Hkv, 1))).astype(np.float32))
    q = rng.standard_normal((B, Hq, 128)) * 2
    for scheme in ("int8_dither", "int8_rtn", "fp8_e4m3", "kivi2", "blackbox"):
        c = OracleCache(1, Hq, Hkv, B, scheme, v_witness=True)
        if scheme == "blackbox":
            c.write(0, K, V, np.round(K * 2) / 2, np.round(V * 2) / 2)
        else:
            c.write(0, K, V)
        r = c.decode(0, q, 1e-2)
        assert np.all(c.wv16[0].astype(np.float64) >= c.wv64[0])
        for i in range(B):
            for j in range(Hq):
                h = j // (Hq // Hkv)
                kh, vh, _, _, _ = c.group_view(0, i, h)
                _, p, _ = meter.attention(q[i, j:j + 1], kh, vh)
                err = np.linalg.norm(p[0] @ (V[i, :, h].astype(np.float64) - vh))
                assert err <= r["meter_v"][i, j] * (1 + 1e-12)
                assert r["meter_v"][i, j] > 0


def test_value_meter_is_tight_for_a_shared_residual():
    """v^_t = v_t - r for every token: the value error is exactly ||r|| whatever the weights, and
    E_V = sum p~ fp16_ru(||r||) = fp16_ru(||r||)."""
    rng = np.random.default_rng(10)
    S = 50
    K = fp.bf16_rn(rng.standard_normal((1, S, 1, 128)).astype(np.float32))
    # multiples of 1/8 below 16 in magnitude: V and V - r are exact in bfloat16
    V = (np.round(np.clip(rng.standard_normal((1, S, 1, 128)), -7, 7) * 8) / 8).astype(np.float32)
    r = np.zeros(128, np.float32)
    r[[3, 70, 100]] = [0.25, -0.5, 0.125]
    c = OracleCache(1, 2, 1, 1, "blackbox", v_witness=True)
    c.write(0, K, V, K, V - r)
    q = rng.standard_normal((1, 2, 128)) * 3
    res = c.decode(0, q, 1e-2)
    norm = math.sqrt(0.25 ** 2 + 0.5 ** 2 + 0.125 ** 2)
    stored = float(fp.fp16_ru(norm * (1 + 2.0 ** -48)))
    for j in range(2):
        kh, vh, _, _, _ = c.group_view(0, 0, 0)
        _, p, _ = meter.attention(q[0, j:j + 1], kh, vh)
        assert abs(np.linalg.norm(p[0] @ (V[0, :, 0].astype(np.float64) - vh)) - norm) < 1e-12
        assert abs(res["meter_v"][0, j] - stored) < 1e-12
    assert stored >= norm and stored <= norm * (1 + 2.0 ** -10)


def test_value_meter_with_uniform_weights_is_the_mean_witness():
    rng = np.random.default_rng(12)
    S = 33
    K = fp.bf16_rn(rng.standard_normal((1, S, 1, 128)).astype(np.float32))
    V = fp.bf16_rn(rng.standard_normal((1, S, 1, 128)).astype(np.float32))
    c = OracleCache(1, 1, 1, 1, "int8_dither", v_witness=True)
    c.write(0, K, V)
    res = c.decode(0, np.zeros((1, 1, 128)), 1e-2)
    assert abs(res["meter_v"][0, 0] - c.wv16[0][0, :, 0].astype(np.float64).mean()) < 1e-12
    # and the witness is the row norm of the residual, over all 128 dims
    assert np.allclose(c.wv64[0][0, :, 0], np.sqrt(((V[0, :, 0] - c.vhat[0][0, :, 0]) ** 2).sum(-1)), rtol=1e-14)
