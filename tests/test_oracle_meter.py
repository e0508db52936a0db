"""Pins of the oracle's decode side: attention, Tier A/B, the TV meter, split merge."""
import math

import numpy as np
import pytest
import scipy.stats as st

from oracle import OracleCache, meter, quant
from workload import WORKLOADS, gen_kv, gen_q


def _tiny_cache(scheme):
    w = WORKLOADS["tiny"].with_(scheme=scheme)
    c = OracleCache(w.n_layers, w.n_q_heads, w.n_kv_heads, w.batch, scheme, w.seed, w.steps)
    K, V = gen_kv(w, 0)
    c.write(0, K, V)
    return w, c


def test_attention_matches_explicit_loops():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((2, 128))
    k = rng.standard_normal((5, 128))
    v = rng.standard_normal((5, 128))
    _, p, out = meter.attention(q, k, v)
    for j in range(2):
        lg = [sum(q[j, c] * k[t, c] for c in range(128)) / math.sqrt(128) for t in range(5)]
        e = [math.exp(x - max(lg)) for x in lg]
        z = sum(e)
        for c in (0, 63, 127):
            assert abs(out[j, c] - sum(e[t] / z * v[t, c] for t in range(5))) < 1e-12


@pytest.mark.parametrize("scheme", ["int8_dither", "fp8_e4m3", "kivi2"])
def test_tv_below_meter_on_every_tiny_cell(scheme):
    """TV(p, p~) <= meter, brute force over every (head, step) of the tiny case, Tier A for all
    schemes and Tier B for the dithered one (its failure probability is delta_loc per cell)."""
    w, c = _tiny_cache(scheme)
    n_checked = 0
    for step in range(w.steps):
        q = gen_q(w, 0, step)
        r = c.decode(0, q, w.delta_req)
        for i in range(w.batch):
            for h in range(w.n_kv_heads):
                js = slice(h * w.group, (h + 1) * w.group)
                _, p, _ = meter.attention(q[i, js], c.k[0][i, :, h], c.v[0][i, :, h])
                _, pt, _ = meter.attention(q[i, js], c.khat[0][i, :, h], c.v[0][i, :, h])
                tv = meter.tv_exact(p, pt)
                assert np.all(tv <= r["meter_a"][i, js] * (1 + 1e-12))
                if scheme == "int8_dither":
                    assert np.all(tv <= r["meter_b"][i, js] * (1 + 1e-12))
                n_checked += tv.size
    assert n_checked == w.steps * w.n_q_heads


def test_meter_closed_forms():
    rng = np.random.default_rng(1)
    pt = meter.softmax(rng.standard_normal((3, 40)))
    # no error -> meter 0 exactly
    assert np.all(meter.tv_meter(pt, np.zeros((3, 40)))[0] == 0)
    # uniform error eps: A = e^eps, meter = (e^{2 eps} - 1)/2
    for eps in (1e-6, 1e-3, 0.1, 0.4):
        m, raw, _ = meter.tv_meter(pt, np.full((3, 40), eps))
        np.testing.assert_allclose(raw, math.expm1(2 * eps) / 2, rtol=1e-12)
    # large error saturates at 1
    assert np.all(meter.tv_meter(pt, np.full((3, 40), 5.0))[0] == 1.0)


def test_meter_is_nearly_tight_for_one_small_mass_token():
    """One token of compressed weight p0 carries error c, all others none: the true TV is
    D/(1+D) - O(p0), the bound D + D^2/2, so the ratio tends to 1 as D -> 0."""
    S = 1000
    lt = np.zeros(S)
    lt[0] = -12.0                                   # small compressed mass on token 0
    pt = meter.softmax(lt[None])
    for Dt in (1e-2, 1e-3):
        c0 = math.log1p(Dt / pt[0, 0])
        l_exact = lt.copy()
        l_exact[0] += c0                            # |l - l~| = c0 on token 0 only
        p = meter.softmax(l_exact[None])
        c = np.zeros((1, S))
        c[0, 0] = c0
        m, raw, Dv = meter.tv_meter(pt, c)
        tv = meter.tv_exact(p, pt)[0]
        assert tv <= raw[0]
        assert tv / raw[0] > 0.985


def test_tier_b_variance_proxy_is_the_logit_error_variance():
    """Dither theory: with q fixed, E[eps_t^2] over dither draws equals
    s2_t = (1/d) sum_c q_c^2 s_c^2 / 12 [WitCert summary, Tier B paragraph]."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal((1, 128)).astype(np.float32)
    x[0, 10] *= 50
    q = rng.standard_normal(128) * 1.5
    n = 20000
    xi = (rng.integers(0, 2 ** 24, size=(n, 128)) * 2.0 ** -24 - 0.5).astype(np.float32)
    X = np.repeat(x, n, 0)
    _, s16, xh, _ = quant.write_int8_dither(X, xi)
    eps = (X.astype(np.float64) - xh) @ q / math.sqrt(128)
    var_pred = meter.tier_b(q[None], s16[:1].astype(np.float64), 1, 1.0)[0, 0] ** 2 / (2 * math.log(2.0))
    assert abs(np.mean(eps ** 2) / var_pred - 1) < 4 * math.sqrt(2 / n)
    # and the exact variance is what the variance proxy names (uniform residual: s^2/12)
    assert abs(np.mean(eps) ) < 4 * math.sqrt(var_pred / n)


def test_tier_b_single_token_tail_matches_gaussian_limit():
    """S = 1: u = sqrt(2 s2 log(2/delta)).  The logit error is a sum of 128 independent uniform
    terms, close to Gaussian, so P(|eps| > u) must be near 2(1 - Phi(sqrt(2 log(2/delta)))),
    a number fixed by the normal law alone; and never above delta."""
    rng = np.random.default_rng(3)
    q = rng.standard_normal(128)
    s = np.full((1, 4), 0.05)
    n = 200000
    r = (rng.uniform(-0.5, 0.5, size=(n, 128)) * 0.05)
    eps = r @ q / math.sqrt(128)
    for delta in (0.5, 0.2):
        u = meter.tier_b(q[None], s, 1, delta)[0, 0]
        rate = np.mean(np.abs(eps) > u)
        gauss = 2 * (1 - st.norm.cdf(math.sqrt(2 * math.log(2 / delta))))
        assert rate <= delta
        assert abs(rate / gauss - 1) < 0.12, (delta, rate, gauss)


def test_tier_b_violation_rate_below_delta_on_nonadaptive_queries():
    """Fresh random queries independent of the dither; delta_loc raised so violations are seen.
    The rate of 'some token of the cell exceeds u_t' must not exceed delta_loc."""
    rng = np.random.default_rng(4)
    S, delta = 256, 0.2
    k = rng.standard_normal((S, 128)).astype(np.float32)
    k[:, 10] *= 20
    trials, viol = 600, 0
    for tr in range(trials):
        xi = (rng.integers(0, 2 ** 24, size=(S, 128)) * 2.0 ** -24 - 0.5).astype(np.float32)
        _, s16, kh, _ = quant.write_int8_dither(k, xi)
        q = rng.standard_normal((1, 128)) * 2
        u = meter.tier_b(q, s16.astype(np.float64), S, delta)[0]
        eps = np.abs((k - kh) @ q[0]) / math.sqrt(128)
        viol += bool(np.any(eps > u))
    upper = st.binom.ppf(0.99, trials, delta) / trials
    assert viol / trials <= upper


def test_delta_loc_uses_query_heads():
    """The pages count 100,352,000 monitored cells for 1000 requests of a 28-layer model with 28
    query heads over 128 steps; that product fixes H in delta_loc = delta_req/(L*H*T) as the
    number of query heads (with the 4 KV heads it would be 14,336,000)."""
    L, Hq, Hkv, T = 28, 28, 4, 128
    assert 1000 * L * Hq * T == 100_352_000
    assert 1000 * L * Hkv * T != 100_352_000
    assert meter.delta_loc(1e-2, L, Hq, T) == pytest.approx(1e-2 / 100_352)


@pytest.mark.parametrize("n_splits", [1, 2, 8, 37])
def test_split_merge_equals_unsplit(n_splits):
    w, c = _tiny_cache("int8_dither")
    q = gen_q(w, 0, 0)[0, :2].astype(np.float64)
    kh, vh, wst, ks, rep = c.group_view(0, 0, 0)
    S = kh.shape[0]
    dl = meter.delta_loc(w.delta_req, 1, w.n_q_heads, w.steps)
    ref = meter.decode_ref(q, kh, vh, wst, ks, rep, dl)
    bounds = np.linspace(0, S, n_splits + 1).astype(int)
    states = [meter.partial_state(q, kh, vh, ref["eps"], ref["u"], a, b) for a, b in zip(bounds[:-1], bounds[1:])]
    mg = meter.merge_states(states)
    np.testing.assert_allclose(mg["out"], ref["out"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(mg["D_a"], ref["D_a"], rtol=1e-12)
    np.testing.assert_allclose(mg["D_b"], ref["D_b"], rtol=1e-12)
    np.testing.assert_allclose(mg["meter_b"], ref["meter_b"], rtol=1e-12)


def test_empty_context_gives_zero_output_and_meters():
    r = meter.decode_ref(np.ones((2, 128)), np.zeros((0, 128)), np.zeros((0, 128)), np.zeros((0, 16)),
                         np.zeros((0, 4)), None, 1e-6)
    assert np.all(r["out"] == 0) and np.all(r["meter_a"] == 0) and np.all(r["meter_b"] == 0)


def test_meters_against_50_digit_arithmetic():
    """Four-way cross-check leg: recompute a few tiny-case meters with 50-digit mpmath."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    w, c = _tiny_cache("int8_dither")
    q = gen_q(w, 0, 1)
    r = c.decode(0, q, w.delta_req)
    kh, _, wst, ks, _ = c.group_view(0, 0, 1)
    S = kh.shape[0]
    dl = mp.mpf(w.delta_req) / (1 * w.n_q_heads * w.steps)
    for j in (2, 3):
        qj = [mp.mpf(float(x)) for x in q[0, j]]
        lg = [mp.fsum(qj[ch] * mp.mpf(float(kh[t, ch])) for ch in range(128)) / mp.sqrt(128) for t in range(S)]
        mx = max(lg)
        e = [mp.exp(x - mx) for x in lg]
        Z = mp.fsum(e)
        qb = [mp.sqrt(mp.fsum(qj[dd] ** 2 for dd in quant.BAND_DIMS[b])) for b in range(16)]
        epsA = [mp.fsum(qb[b] * mp.mpf(float(wst[t, b])) for b in range(16)) / mp.sqrt(128) for t in range(S)]
        qg = [mp.fsum(qj[ch] ** 2 for ch in range(32 * gg, 32 * gg + 32)) for gg in range(4)]
        u = [mp.sqrt(2 * mp.fsum(qg[gg] * mp.mpf(float(ks[t, gg])) ** 2 for gg in range(4)) / (12 * 128)
                     * mp.log(2 * S / dl)) for t in range(S)]
        for cvec, key in ((epsA, "raw_a"), (u, "raw_b")):
            A = mp.fsum(e[t] / Z * mp.exp(cvec[t]) for t in range(S))
            raw = (A * A - 1) / 2
            assert abs(float(raw) / r[key][0, j] - 1) < 1e-10


@pytest.mark.parametrize("scheme", ["fp8_e4m3", "int8_dither"])
@pytest.mark.parametrize("S", [256, 16 * 9 + 5])
def test_block_risk_is_each_blocks_share_of_the_gate_tier(scheme, S):
    """Block risks R_blk = sum_{t in blk} p~_t expm1(c_t): a brute force over tokens with
    explicit loops, and their sum over the blocks (ragged tail included) equals D of the gate's
    tier: Tier B for the dithered scheme, Tier A otherwise."""
    w = WORKLOADS["tiny"].with_(scheme=scheme, context=S)
    c = OracleCache(w.n_layers, w.n_q_heads, w.n_kv_heads, w.batch, scheme, w.seed, w.steps)
    K, V = gen_kv(w, 0)
    c.write(0, K, V)
    q = gen_q(w, 0, 0)
    kh, vh, wst, ks, rep = c.group_view(0, 0, 1)
    dl = meter.delta_loc(w.delta_req, w.n_layers, w.n_q_heads, w.steps)
    r = meter.decode_ref(q[0, 2:4], kh, vh, wst, ks, rep, dl)
    cg = r["u"] if scheme == "int8_dither" else r["eps"]
    D = r["D_b"] if scheme == "int8_dither" else r["D_a"]
    nblk = (S + 15) // 16
    assert r["risk"].shape == (2, nblk)
    for j in range(2):
        for b in range(nblk):
            want = 0.0
            for t in range(16 * b, min(16 * b + 16, S)):
                want += r["p"][j, t] * math.expm1(cg[j, t])
            assert abs(r["risk"][j, b] - want) <= 1e-12 * max(want, 1e-300)
        assert abs(math.fsum(r["risk"][j]) - D[j]) <= 1e-12 * D[j]
    # the two tiers differ on the dithered scheme, so the identity picks out the tier
    if scheme == "int8_dither":
        assert np.all(np.abs(r["D_a"] - r["D_b"]) > 1e-6 * r["D_b"])
