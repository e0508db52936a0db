"""Shared helpers of the GPU parity tests: run a workload through the library and the oracle."""
from __future__ import annotations

import numpy as np
import torch

import kv_cache_quantization_witcert_gb300 as wc
from kv_cache_quantization_witcert_gb300 import _lib
from oracle import OracleCache, meter, quant
from oracle.philox import dither

# Meters: GPU >= oracle with no relative slack (the library rounds every meter up) and
# GPU <= oracle * (1 + 1e-4); a GPU NaN where the oracle has a number fails.  The one absolute
# allowance, 2^-99, is for values below fp32's range: the meters are fp32, terms whose weights
# fall under 2^-126 are dropped, and the library adds 2^-100 to every positive meter and risk.
METER_REL = 1e-4
METER_ABS = 2.0 ** -99


def torch_dtype(w):
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def to_dev(x, w):
    return torch.from_numpy(np.ascontiguousarray(x)).to(device="cuda").to(torch_dtype(w))


def make_pair(w, scheme=None, n_splits=None, extra_tokens=None, gate_blocks=0, v_witness=False, max_pages=0):
    scheme = scheme or w.scheme
    cap = w.context + (w.steps if extra_tokens is None else extra_tokens)
    gpu = wc.Cache(w.n_layers, w.n_q_heads, w.n_kv_heads, w.batch, cap, scheme, dtype=torch_dtype(w),
                   seed=w.seed, total_steps=w.steps, n_splits=w.n_splits if n_splits is None else n_splits,
                   max_repair_blocks=gate_blocks, v_witness=v_witness, max_pages=max_pages)
    ref = OracleCache(w.n_layers, w.n_q_heads, w.n_kv_heads, w.batch, scheme, w.seed, w.steps, v_witness=v_witness)
    return gpu, ref


def tensor_function(x, seed=0):
    """A caller's quantize-dequantize function for the black-box scheme (test input): keep five
    mantissa bits, and move 1% of the entries by a seeded N(0, 1) amount."""
    x = np.asarray(x, np.float32)
    m, e = np.frexp(x)
    y = np.ldexp(np.trunc(m * 32.0) / 32.0, e).astype(np.float32)
    rng = np.random.default_rng(seed)
    mask = rng.random(x.shape) < 0.01
    y[mask] += rng.standard_normal(int(mask.sum())).astype(np.float32)
    return y


def write_both(gpu, ref, layer, K, V, w, seed=0):
    """Append K, V to both caches; the black-box scheme also gets f(K), f(V), and the oracle gets
    exactly the values the device received."""
    if ref.scheme != "blackbox":
        gpu.witcert_write(layer, to_dev(K, w), to_dev(V, w))
        ref.write(layer, K, V)
        return
    kh = to_dev(tensor_function(K, seed), w)
    vh = to_dev(tensor_function(V, seed + 1), w)
    gpu.witcert_write_hat(layer, to_dev(K, w), to_dev(V, w), kh, vh)
    ref.write(layer, K, V, kh.float().cpu().numpy(), vh.float().cpu().numpy())


def check_meter(gpu, ref, rel=METER_REL, what="", raw=False):
    """GPU values never below the oracle's (up to METER_ABS) and within rel above them.

    raw=True: the values are raw meters D + D^2/2.  Where the oracle's exceeds 1, the meter
    min(1, D + D^2/2) is 1 on both sides, and the tolerance above applies to
    D = sqrt(1 + 2 raw) - 1, the sum the gate compares with D*: the raw value's relative
    excess is up to twice D's there."""
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    low = g < r - METER_ABS
    high = g > r * (1 + rel) + METER_ABS
    if raw:
        with np.errstate(invalid="ignore", over="ignore"):
            big = r > 1
            dg, dr = np.sqrt(1 + 2 * g) - 1, np.sqrt(1 + 2 * r) - 1
            high = np.where(big, dg > dr * (1 + rel) + METER_ABS, high)
    nan = np.isnan(g) & ~np.isnan(r)          # a NaN bounds nothing and fails both comparisons
    if low.any() or high.any() or nan.any():
        idx = np.argwhere(low | high | nan)[:5]
        detail = [(tuple(ix), g[tuple(ix)], r[tuple(ix)]) for ix in idx]
        raise AssertionError(f"{what}: {low.sum()} below, {high.sum()} above tolerance, {nan.sum()} NaN: {detail}")


def check_write(gpu, ref, layer, scheme):
    """Codes and scales bit-exact; stored witness bit-exact and bracketing the float64 norm."""
    S = ref.length(layer)
    if scheme == "blackbox":     # the stored bf16 values are the oracle's bf16(f(x)), bit for bit
        kc = gpu.export(layer, _lib.X_K_CODES).float().cpu().numpy().astype(np.float64)
        vc = gpu.export(layer, _lib.X_V_CODES).float().cpu().numpy().astype(np.float64)
        np.testing.assert_array_equal(kc, ref.khat[layer])
        np.testing.assert_array_equal(vc, ref.vhat[layer])
    else:
        kc = gpu.export(layer, _lib.X_K_CODES).cpu().numpy()
        vc = gpu.export(layer, _lib.X_V_CODES).cpu().numpy()
    if scheme in ("int8_dither", "int8_rtn"):
        np.testing.assert_array_equal(kc.view(np.int8).astype(np.int16), ref.kcode[layer])
        np.testing.assert_array_equal(vc.view(np.int8).astype(np.int16), ref.vcode[layer])
        ks = gpu.export(layer, _lib.X_K_SCALES).cpu().numpy()
        vs = gpu.export(layer, _lib.X_V_SCALES).cpu().numpy()
        np.testing.assert_array_equal(ks.view(np.uint16), ref.kscale[layer].view(np.uint16))
        np.testing.assert_array_equal(vs.view(np.uint16), ref.vscale[layer].view(np.uint16))
    elif scheme == "fp8_e4m3":
        np.testing.assert_array_equal(kc.astype(np.int16), ref.kcode[layer])
        np.testing.assert_array_equal(vc.astype(np.int16), ref.vcode[layer])
    elif scheme == "kivi2":
        full = (S // 16) * 16
        np.testing.assert_array_equal(kc[:, :full].astype(np.int16), ref.kcode[layer][:, :full])
        np.testing.assert_array_equal(vc.astype(np.int16), ref.vcode[layer])
        vs = gpu.export(layer, _lib.X_V_SCALES).cpu().numpy()
        vz = gpu.export(layer, _lib.X_V_ZEROS).cpu().numpy()
        np.testing.assert_array_equal(vs.view(np.uint16), ref.vscale[layer].view(np.uint16))
        np.testing.assert_array_equal(vz.view(np.uint16), ref.vzero[layer].view(np.uint16))
        ksc = gpu.export(layer, _lib.X_KIVI_K_SCALE).cpu().numpy()
        kzr = gpu.export(layer, _lib.X_KIVI_K_ZERO).cpu().numpy()
        for (i, h, b), (s, z) in ref.kivi_kp[layer].items():
            np.testing.assert_array_equal(ksc[i, b, h].view(np.uint16), s.view(np.uint16))
            np.testing.assert_array_equal(kzr[i, b, h].view(np.uint16), z.view(np.uint16))
    w = gpu.export(layer, _lib.X_WITNESS).cpu().numpy()
    np.testing.assert_array_equal(w.view(np.uint16), ref.w16[layer].view(np.uint16))
    w64 = ref.w64[layer]
    wg = w.astype(np.float64)
    assert np.all(wg >= w64)
    # above fp16's largest value the rounded-up witness is +inf
    assert np.all((wg <= np.maximum(w64 * (1 + 1e-3), w64 + 2.0 ** -24)) | (np.isinf(wg) & (w64 > 65504.0)))
    if ref.v_witness:
        wv = gpu.export(layer, _lib.X_V_WITNESS).cpu().numpy()
        np.testing.assert_array_equal(wv.view(np.uint16), ref.wv16[layer].view(np.uint16))
        wvg, wv64 = wv.astype(np.float64), ref.wv64[layer]
        assert np.all(wvg >= wv64)
        assert np.all((wvg <= np.maximum(wv64 * (1 + 1e-3), wv64 + 2.0 ** -24)) | (np.isinf(wvg) & (wv64 > 65504.0)))
    return w


def check_decode(gpu, ref, layer, q_host, w, delta_req, rel=METER_REL):
    """Decode both sides on the same query; the oracle uses the GPU's stored witness."""
    out, m = gpu.decode(layer, to_dev(q_host, w), delta_req)
    ref.w16[layer] = gpu.export(layer, _lib.X_WITNESS).cpu().numpy()
    if ref.v_witness:
        ref.wv16[layer] = gpu.export(layer, _lib.X_V_WITNESS).cpu().numpy()
    r = ref.decode(layer, q_host, delta_req)
    o = out.cpu().numpy().astype(np.float64)
    g = ref.g
    for i in range(ref.B):
        for h in range(ref.Hkv):
            vmax = np.abs(ref.v[layer][i, :, h]).max() if ref.length(layer) else 1.0
            d = np.abs(o[i, h * g:(h + 1) * g] - r["out"][i, h * g:(h + 1) * g]).max()
            assert d <= 2e-3 * vmax, f"out seq {i} head {h}: {d} > {2e-3 * vmax}"
    check_meter(m["raw_a"].cpu().numpy(), r["raw_a"], rel, "raw_a", raw=True)
    check_meter(m["meter_a"].cpu().numpy(), r["meter_a"], rel, "meter_a")
    if ref.scheme == "int8_dither":
        check_meter(m["raw_b"].cpu().numpy(), r["raw_b"], rel, "raw_b", raw=True)
        check_meter(m["meter_b"].cpu().numpy(), r["meter_b"], rel, "meter_b")
    else:
        assert np.all(np.isnan(m["meter_b"].cpu().numpy()))
    if ref.v_witness:
        check_meter(m["meter_v"].cpu().numpy(), r["meter_v"], rel, "meter_v")
    return out, m, r


def oracle_group(w, layer, K, V, q, i, h, scheme, dloc, k_pos0=0):
    """Oracle decode of one (sequence, KV head) group straight from K/V [S, d] (for sampled cells)."""
    S = K.shape[0]
    pos = np.arange(k_pos0, k_pos0 + S)
    if scheme == "int8_dither":
        _, ks, kh, _ = quant.write_int8_dither(K, dither(w.seed, layer, h, pos, 0))
        _, _, vh, _ = quant.write_int8_dither(V, dither(w.seed, layer, h, pos, 1))
        kscales = ks.astype(np.float64)
    elif scheme == "fp8_e4m3":
        _, kh = quant.write_fp8(K)
        _, vh = quant.write_fp8(V)
        kscales = None
    else:
        kh = K.astype(np.float64).copy()
        for b in range(S // 16):
            kh[16 * b:16 * b + 16] = quant.write_kivi2_k(K[16 * b:16 * b + 16])[3]
        vh = quant.write_kivi2_v(V)[3]
        kscales = None
    wst = quant.witness_stored(quant.witness(K - kh)).astype(np.float64)
    return meter.decode_ref(q, kh, vh, wst, kscales, None, dloc)


# Block risks: as the meters, GPU >= oracle and <= oracle * (1 + 1e-4) up to METER_ABS.
RISK_ABS = METER_ABS


def check_risk(gpu, ref, rel=METER_REL, what="risk"):
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    low = g < r - RISK_ABS
    high = g > r * (1 + rel) + RISK_ABS
    nan = np.isnan(g)
    if low.any() or high.any() or nan.any():
        idx = np.argwhere(low | high | nan)[:5]
        detail = [(tuple(ix), g[tuple(ix)], r[tuple(ix)]) for ix in idx]
        raise AssertionError(f"{what}: {low.sum()} below, {high.sum()} above tolerance, {nan.sum()} NaN: {detail}")


def gate_tie_zone(risk_row, repaired, tau, rel=METER_REL):
    """True when the oracle's decision for one cell could change under a relative change of
    `rel` in its risks: its total, or the remaining risk just before or after its cut, within
    rel of D*, or the last taken and first untaken blocks within rel of each other."""
    import math
    from oracle.gate import canonical_risk, d_star, select_cell
    r = [canonical_risk(x) for x in np.asarray(risk_row, np.float32)]
    cand = [b for b in range(len(r)) if not repaired[b]]
    order = sorted(cand, key=lambda b: (-r[b], b))
    ds = d_star(tau)
    near = lambda x: abs(x - ds) <= rel * max(ds, x)
    if near(math.fsum(r[b] for b in cand)):
        return True
    k = len(select_cell(risk_row, repaired, tau))
    if k == 0:
        return False
    rem = math.fsum(r[b] for b in order[k:])
    if near(rem) or near(rem + r[order[k - 1]]):
        return True
    return k < len(order) and abs(r[order[k - 1]] - r[order[k]]) <= rel * r[order[k - 1]]


def check_gate_end_to_end(oracle_risk, repaired_before, tau, gpu_repaired_after, g):
    """The oracle gate fed the oracle's OWN risks [B, Hq, nblk] must pick exactly the blocks
    the GPU repaired, outside the tie zone; returns the number of tie-zone cells (expected 0)."""
    from oracle.gate import select_cell
    B, Hq, nblk = oracle_risk.shape
    ties = 0
    for i in range(B):
        for h in range(Hq // g):
            want = np.asarray(repaired_before[i, h, :nblk], bool).copy()
            tie = False
            for j in range(h * g, (h + 1) * g):
                if gate_tie_zone(oracle_risk[i, j], repaired_before[i, h, :nblk], tau):
                    tie = True
                for b in select_cell(oracle_risk[i, j], repaired_before[i, h, :nblk], tau):
                    want[b] = True
            if tie:
                ties += 1
                continue
            np.testing.assert_array_equal(np.asarray(gpu_repaired_after[i, h, :nblk], bool), want,
                                          err_msg=f"end-to-end gate, sequence {i} KV head {h}")
    return ties
