"""Parity at the full sizes of the long-context workloads, on sampled outputs.

Long-context sweep points (Mistral-7B and Yi-1.5-6B shaped) at 32768 tokens and at the
sweep's longest context, 131072 tokens, and the gated-repair workload (Qwen2.5-7B shaped, batch 8 x 32768, raw-cast FP8 with the gate) are run at
their full batch, head and context sizes, one layer each: a layer's launch configuration
(split count, CTAs, sequences per CTA) depends on the batch, heads and context, not on the
layer count.  Sampled (sequence, KV head) groups are checked against the oracle computed
for those groups alone; the gate's decisions are checked for every group, by the oracle's
gate fed the GPU's block risks.
"""
import numpy as np
import pytest
import torch

import kv_cache_quantization_witcert_gb300 as wc
from kv_cache_quantization_witcert_gb300 import _lib
from oracle import meter, quant
from oracle.philox import dither
from oracle.gate import gate_group
from workload import WORKLOADS, gen_kv, gen_q, sweep_workload

from gpu_helpers import check_gate_end_to_end, check_meter, check_risk, oracle_group, to_dev

pytestmark = pytest.mark.gpu

LONG = 32768


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    wc.load()


def check_group(w, o, m, r, i, h, V, tier_b):
    js = slice(h * w.group, (h + 1) * w.group)
    vmax = np.abs(V[i, :, h]).max()
    d = np.abs(o[i, js] - r["out"]).max()
    assert d <= 2e-3 * vmax, f"out seq {i} head {h}: {d} > {2e-3 * vmax}"
    check_meter(m["raw_a"].cpu().numpy()[i, js], r["raw_a"], what=f"raw_a seq {i} head {h}", raw=True)
    check_meter(m["meter_a"].cpu().numpy()[i, js], r["meter_a"], what=f"meter_a seq {i} head {h}")
    if tier_b:
        check_meter(m["raw_b"].cpu().numpy()[i, js], r["raw_b"], what=f"raw_b seq {i} head {h}", raw=True)


@pytest.mark.parametrize("model,batch,scheme,context", [("mistral", 16, "int8_dither", LONG), ("yi", 8, "fp8_e4m3", LONG),
                                                         ("mistral", 1, "int8_dither", 4 * LONG)])
def test_long_context_sweep_point_sampled_groups(model, batch, scheme, context):
    """One layer of a sweep point (the bench sweeps four), automatic split count: two 32768-token
    points and the sweep's longest context, 131072 tokens, for one sequence."""
    w = sweep_workload(model, batch, context, scheme, n_layers=4)
    gpu = wc.Cache(w.n_layers, w.n_q_heads, w.n_kv_heads, w.batch, w.context + 1, scheme, dtype=torch.bfloat16,
                   seed=w.seed, total_steps=w.steps)
    dl = meter.delta_loc(w.delta_req, w.n_layers, w.n_q_heads, w.steps)
    K, V = gen_kv(w, 0)
    gpu.witcert_write(0, to_dev(K, w), to_dev(V, w))
    q = gen_q(w, 0, 0)
    out, m = gpu.decode(0, to_dev(q, w), w.delta_req)
    o = out.cpu().numpy()
    for i, h in [(0, 0), (batch - 1, w.n_kv_heads - 1), (batch // 2, 1)]:
        js = slice(h * w.group, (h + 1) * w.group)
        r = oracle_group(w, 0, K[i, :, h], V[i, :, h], q[i, js], i, h, scheme, dl)
        check_group(w, o, m, r, i, h, V, scheme == "int8_dither")
    assert gpu.witcert_stats()["device_errors"] == 0
    gpu.close()


def oracle_fp8_repaired(K, V, q, rep_blocks):
    """Oracle decode of one FP8 group whose listed blocks hold exact keys and zero witnesses."""
    _, kh = quant.write_fp8(K)
    _, vh = quant.write_fp8(V)
    wst = quant.witness_stored(quant.witness(K - kh)).astype(np.float64)
    rep = np.zeros(K.shape[0], bool)
    for b in rep_blocks:
        rep[16 * b:16 * b + 16] = True
    kh = kh.copy()
    kh[rep] = K[rep]
    wst[rep] = 0.0
    return meter.decode_ref(q, kh, vh, wst, None, rep, None)


def test_gated_config_full_size_gate_decisions_and_repaired_decode():
    """Gated workload at full size (batch 8 x 32768, 28q/4kv, raw-cast FP8), one layer: every
    group's pages-in equal the oracle gate's choice from the GPU's risks at tau = 0.5, and the
    next decode matches the oracle on the repaired groups."""
    w = WORKLOADS["gated"].with_(n_layers=1)
    nblk = w.context // 16
    pool = w.batch * w.n_kv_heads * (nblk + 1)
    gpu = wc.Cache(1, w.n_q_heads, w.n_kv_heads, w.batch, w.context + 1, "fp8_e4m3", dtype=torch.bfloat16,
                   seed=w.seed, total_steps=w.steps, max_repair_blocks=pool)
    K, V = gen_kv(w, 0)
    gpu.witcert_write(0, to_dev(K, w), to_dev(V, w))
    q = gen_q(w, 0, 0)
    out, m = gpu.decode(0, to_dev(q, w), w.delta_req)
    o = out.cpu().numpy()
    sampled = [(0, 0), (w.batch - 1, w.n_kv_heads - 1)]
    for i, h in sampled:
        js = slice(h * w.group, (h + 1) * w.group)
        r = oracle_group(w, 0, K[i, :, h], V[i, :, h], q[i, js], i, h, "fp8_e4m3", None)
        check_group(w, o, m, r, i, h, V, False)
    risk = gpu.export(0, _lib.X_BLOCK_RISK).cpu().numpy()
    assert risk.shape == (w.batch, w.n_q_heads, nblk)
    tau = 0.5
    gpu.witcert_gate(0, tau)
    slots = gpu.export(0, _lib.X_SLOTS).cpu().numpy()
    picked = {}
    for i in range(w.batch):
        for h in range(w.n_kv_heads):
            js = slice(h * w.group, (h + 1) * w.group)
            sel = gate_group(risk[i, js], np.zeros(nblk, bool), tau)
            want = np.zeros(nblk, bool)
            want[sel] = True
            np.testing.assert_array_equal(slots[i, h] >= 0, want, err_msg=f"seq {i} head {h}")
            picked[(i, h)] = sel
    st = gpu.witcert_gate_stats()
    total = sum(len(s) for s in picked.values())
    assert st["blocks_paged_in"] == total > 0 and st["blocks_dropped"] == 0
    q2 = gen_q(w, 0, 1)
    out2, m2 = gpu.decode(0, to_dev(q2, w), w.delta_req)
    o2 = out2.cpu().numpy()
    for i, h in sampled:
        js = slice(h * w.group, (h + 1) * w.group)
        r = oracle_fp8_repaired(K[i, :, h], V[i, :, h], q2[i, js], picked[(i, h)])
        check_group(w, o2, m2, r, i, h, V, False)
    assert gpu.witcert_stats()["device_errors"] == 0
    gpu.close()


def test_gated_config_full_size_int8_dither_gate():
    """The gated workload's shape (batch 8 x 32768, 28q/4kv) on a dithered INT8 cache with the
    gate, one layer: the Tier B block risks of sampled groups match the oracle's (never below,
    within 1e-4); every group's pages-in equal the oracle gate's choice from the GPU's risks at
    tau = 4; for the sampled groups the oracle gate fed the oracle's own risks picks the same
    blocks (tie zone empty); the repaired decode matches the oracle."""
    w = WORKLOADS["gated"].with_(n_layers=1, scheme="int8_dither")
    nblk = w.context // 16
    pool = w.batch * w.n_kv_heads * (nblk + 1)
    gpu = wc.Cache(1, w.n_q_heads, w.n_kv_heads, w.batch, w.context + 1, "int8_dither", dtype=torch.bfloat16,
                   seed=w.seed, total_steps=w.steps, max_repair_blocks=pool)
    K, V = gen_kv(w, 0)
    gpu.witcert_write(0, to_dev(K, w), to_dev(V, w))
    q = gen_q(w, 0, 0)
    dl = meter.delta_loc(w.delta_req, w.n_layers, w.n_q_heads, w.steps)
    out, m = gpu.decode(0, to_dev(q, w), w.delta_req)
    o = out.cpu().numpy()
    risk = gpu.export(0, _lib.X_BLOCK_RISK).cpu().numpy()
    tau = 4.0
    sampled = [(0, 0), (3, 2), (w.batch - 1, w.n_kv_heads - 1)]
    oracle_risk = {}
    for i, h in sampled:
        js = slice(h * w.group, (h + 1) * w.group)
        r = oracle_group(w, 0, K[i, :, h], V[i, :, h], q[i, js], i, h, "int8_dither", dl)
        check_group(w, o, m, r, i, h, V, True)
        check_risk(risk[i, js], r["risk"], what=f"block risk seq {i} head {h}")
        oracle_risk[(i, h)] = r["risk"]
    gpu.witcert_gate(0, tau)
    slots = gpu.export(0, _lib.X_SLOTS).cpu().numpy()
    picked = {}
    for i in range(w.batch):
        for h in range(w.n_kv_heads):
            js = slice(h * w.group, (h + 1) * w.group)
            sel = gate_group(risk[i, js], np.zeros(nblk, bool), tau)
            want = np.zeros(nblk, bool)
            want[sel] = True
            np.testing.assert_array_equal(slots[i, h] >= 0, want, err_msg=f"seq {i} head {h}")
            picked[(i, h)] = sel
    for (i, h), r_own in oracle_risk.items():
        ties = check_gate_end_to_end(r_own[None], np.zeros((1, 1, nblk), bool), tau, (slots[i, h] >= 0)[None, None],
                                     w.group)
        assert ties == 0, f"seq {i} head {h}: {ties} cell groups in the tie zone"
    st = gpu.witcert_gate_stats()
    assert st["blocks_paged_in"] == sum(len(s) for s in picked.values()) > 0 and st["blocks_dropped"] == 0
    q2 = gen_q(w, 0, 1)
    out2, m2 = gpu.decode(0, to_dev(q2, w), w.delta_req)
    o2 = out2.cpu().numpy()
    for i, h in sampled[:2]:
        js = slice(h * w.group, (h + 1) * w.group)
        r = oracle_int8_repaired(w, K[i, :, h], V[i, :, h], q2[i, js], h, picked[(i, h)], dl)
        check_group(w, o2, m2, r, i, h, V, True)
    assert gpu.witcert_stats()["device_errors"] == 0
    gpu.close()


def oracle_int8_repaired(w, K, V, q, h, rep_blocks, dl):
    """Oracle decode of one dithered INT8 group whose listed blocks hold exact keys, zero
    witnesses and no Tier B term."""
    S = K.shape[0]
    pos = np.arange(S)
    _, ks, kh, _ = quant.write_int8_dither(K, dither(w.seed, 0, h, pos, 0))
    _, _, vh, _ = quant.write_int8_dither(V, dither(w.seed, 0, h, pos, 1))
    wst = quant.witness_stored(quant.witness(K - kh)).astype(np.float64)
    rep = np.zeros(S, bool)
    for b in rep_blocks:
        rep[16 * b:16 * b + 16] = True
    kh = kh.copy()
    kh[rep] = K[rep]
    wst[rep] = 0.0
    return meter.decode_ref(q, kh, vh, wst, ks.astype(np.float64), rep, dl)
