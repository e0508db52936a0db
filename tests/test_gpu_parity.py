"""GPU parity through the C ABI against the float64 oracle (needs a GB300)."""
import numpy as np
import pytest
import torch

import kv_cache_quantization_witcert_gb300 as wc
from kv_cache_quantization_witcert_gb300 import _lib
from oracle import meter
from oracle.philox import dither
from workload import WORKLOADS, gen_append_kv, gen_kv, gen_q

from gpu_helpers import (check_decode, check_gate_end_to_end, check_meter, check_risk, check_write, make_pair,
                         oracle_group, to_dev, write_both)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    wc.load()


def test_dither_stream_bit_exact():
    for seed, layer, h, t0, tensor in [(0, 0, 0, 0, 0), (12345678901234, 27, 3, 4090, 1), (2 ** 64 - 1, 5, 7, 131000, 0)]:
        g = wc.witcert_dither(seed, layer, h, t0, 40, tensor).cpu().numpy()
        np.testing.assert_array_equal(g, dither(seed, layer, h, np.arange(t0, t0 + 40), tensor))


@pytest.mark.parametrize("n_splits", [0, 1, 2, 8, 37])
def test_tiny_write_and_metered_decode_with_appends(n_splits):
    w = WORKLOADS["tiny"]
    gpu, ref = make_pair(w, n_splits=n_splits)
    K, V = gen_kv(w, 0)
    gpu.witcert_write(0, to_dev(K, w), to_dev(V, w))
    ref.write(0, K, V)
    wst = check_write(gpu, ref, 0, w.scheme)
    for step in range(w.steps):
        check_decode(gpu, ref, 0, gen_q(w, 0, step), w, w.delta_req)
        k1, v1 = gen_append_kv(w, 0, step)
        gpu.witcert_write(0, to_dev(k1, w), to_dev(v1, w))
        ref.write(0, k1, v1)
    check_write(gpu, ref, 0, w.scheme)
    check_decode(gpu, ref, 0, gen_q(w, 0, w.steps), w, w.delta_req)
    st = gpu.witcert_stats()
    assert st["int8_clamps"] == 0 and st["device_errors"] == 0


ALL_SCHEMES = ["int8_dither", "fp8_e4m3", "kivi2", "int8_rtn", "blackbox"]


@pytest.mark.parametrize("v_witness", [False, True])
@pytest.mark.parametrize("scheme", ALL_SCHEMES)
def test_qwen_shaped_bf16_ragged(scheme, v_witness):
    """28q/4kv, bf16, planted keys and x50 outliers; 3 sequences (a partial sequence group),
    1000 tokens (several splits and a ragged 8-token tail), two steps with an append; with and
    without value witnesses (value meter E_V)."""
    w = WORKLOADS["qwen_1l"].with_(batch=3, context=1000, steps=2, scheme=scheme)
    gpu, ref = make_pair(w, v_witness=v_witness)
    K, V = gen_kv(w, 0)
    write_both(gpu, ref, 0, K, V, w)
    check_write(gpu, ref, 0, scheme)
    check_decode(gpu, ref, 0, gen_q(w, 0, 0), w, w.delta_req)
    k1, v1 = gen_append_kv(w, 0, 0)
    write_both(gpu, ref, 0, k1, v1, w, seed=5)
    check_write(gpu, ref, 0, scheme)
    check_decode(gpu, ref, 0, gen_q(w, 0, 1), w, 1e-3)


@pytest.mark.parametrize("n_splits", [0, 3])
def test_tiny_blackbox_fp32_with_appends_and_value_witness(n_splits):
    """fp32 keys and function outputs (rounded to bf16 by the cache), sixteen single-token appends
    across a block boundary, value witnesses on."""
    w = WORKLOADS["tiny"].with_(scheme="blackbox", steps=16)
    gpu, ref = make_pair(w, n_splits=n_splits, v_witness=True)
    K, V = gen_kv(w, 0)
    write_both(gpu, ref, 0, K, V, w)
    check_write(gpu, ref, 0, "blackbox")
    for step in range(w.steps):
        k1, v1 = gen_append_kv(w, 0, step)
        write_both(gpu, ref, 0, k1, v1, w, seed=100 + step)
        if step % 4 == 3:
            check_write(gpu, ref, 0, "blackbox")
            check_decode(gpu, ref, 0, gen_q(w, 0, step), w, w.delta_req)
    assert gpu.witcert_stats()["device_errors"] == 0


def test_blackbox_identity_function_is_plain_attention():
    """f = identity: zero witnesses and meters, and the output is softmax attention on the exact
    bf16 keys and values."""
    w = WORKLOADS["qwen_1l"].with_(batch=2, context=300, scheme="blackbox")
    gpu, _ = make_pair(w, v_witness=True)
    K, V = gen_kv(w, 0)
    Kd, Vd = to_dev(K, w), to_dev(V, w)
    gpu.witcert_write_hat(0, Kd, Vd, Kd, Vd)
    q = gen_q(w, 0, 0)
    out, m = gpu.decode(0, to_dev(q, w), w.delta_req)
    assert torch.count_nonzero(gpu.export(0, _lib.X_WITNESS)) == 0
    for k in ("meter_a", "raw_a", "meter_v"):
        assert torch.count_nonzero(m[k]) == 0
    o = out.cpu().numpy()
    for i in range(2):
        for j in range(w.n_q_heads):
            _, _, ref = meter.attention(q[i, j:j + 1], K[i, :, j // w.group], V[i, :, j // w.group])
            assert np.abs(o[i, j] - ref[0]).max() <= 2e-3 * np.abs(V[i, :, j // w.group]).max()


def test_write_entry_points_match_the_scheme():
    w = WORKLOADS["tiny"]
    bb, _ = make_pair(w, scheme="blackbox")
    K, V = gen_kv(w, 0)
    with pytest.raises(wc.WitcertError) as e:
        bb.witcert_write(0, to_dev(K, w), to_dev(V, w))
    assert e.value.status == _lib.EINVAL
    i8, _ = make_pair(w)
    with pytest.raises(wc.WitcertError) as e:
        i8.witcert_write_hat(0, to_dev(K, w), to_dev(V, w), to_dev(K, w), to_dev(V, w))
    assert e.value.status == _lib.EINVAL
    i8.witcert_write(0, to_dev(K, w), to_dev(V, w))
    out = torch.empty((w.batch, w.n_q_heads, 128), dtype=torch.float32, device="cuda")
    mv = torch.empty((w.batch, w.n_q_heads), dtype=torch.float32, device="cuda")
    with pytest.raises(wc.WitcertError) as e:     # no value witnesses in this cache
        i8.witcert_decode(0, to_dev(gen_q(w, 0, 0), w), w.delta_req, out, meter_v=mv)
    assert e.value.status == _lib.EINVAL


@pytest.mark.parametrize("scheme", ["int8_dither", "kivi2"])
def test_more_split_ctas_than_the_gpu_holds(scheme):
    """300 splits x 4 KV heads: several waves of split CTAs and 300 partial records per cell
    to merge; results still match the oracle."""
    w = WORKLOADS["qwen_1l"].with_(batch=3, context=1000, steps=1, scheme=scheme)
    gpu, ref = make_pair(w, n_splits=300)
    K, V = gen_kv(w, 0)
    gpu.witcert_write(0, to_dev(K, w), to_dev(V, w))
    ref.write(0, K, V)
    check_decode(gpu, ref, 0, gen_q(w, 0, 0), w, w.delta_req)
    assert gpu.witcert_stats()["device_errors"] == 0


@pytest.mark.parametrize("scheme", ALL_SCHEMES)
def test_kivi_and_all_schemes_across_block_boundaries(scheme):
    """Appends one token at a time across two 16-token boundaries (KIVI closes blocks); value
    witnesses on."""
    w = WORKLOADS["tiny"].with_(context=29, steps=20, scheme=scheme, batch=2)
    gpu, ref = make_pair(w, v_witness=True)
    K, V = gen_kv(w, 0)
    write_both(gpu, ref, 0, K, V, w)
    for step in range(w.steps):
        k1, v1 = gen_append_kv(w, 0, step)
        write_both(gpu, ref, 0, k1, v1, w, seed=7 + step)
        if step % 5 == 4:
            check_write(gpu, ref, 0, scheme)
            check_decode(gpu, ref, 0, gen_q(w, 0, step), w, w.delta_req)


@pytest.mark.parametrize("scheme", ALL_SCHEMES)
def test_meter_off_output_is_bit_identical(scheme):
    w = WORKLOADS["qwen_1l"].with_(batch=5, context=700, scheme=scheme)
    gpu, ref = make_pair(w, v_witness=True)
    K, V = gen_kv(w, 0)
    write_both(gpu, ref, 0, K, V, w)
    q = to_dev(gen_q(w, 0, 0), w)
    on, _ = gpu.decode(0, q, w.delta_req, meters=True)
    off, _ = gpu.decode(0, q, w.delta_req, meters=False)
    assert torch.equal(on, off)


def test_split_invariance_on_gpu():
    w = WORKLOADS["qwen_1l"].with_(batch=2, context=2000)
    K, V = gen_kv(w, 0)
    q = gen_q(w, 0, 0)
    outs = []
    for ns in (1, 2, 8, 37):
        gpu, _ = make_pair(w, n_splits=ns)
        gpu.witcert_write(0, to_dev(K, w), to_dev(V, w))
        outs.append(gpu.decode(0, to_dev(q, w), w.delta_req))
    # P enters the P.V product as fp16 relative to each split's running max, so outputs of
    # different split counts agree to the output bar (2e-3 max|V|), not bitwise; meters are
    # summed in fp32 and agree far inside their 1e-4 bar
    vmax = np.abs(V).max()
    for o, m in outs[1:]:
        np.testing.assert_allclose(o.cpu().numpy(), outs[0][0].cpu().numpy(), atol=2e-3 * vmax, rtol=0)
        for k in ("raw_a", "raw_b"):
            np.testing.assert_allclose(m[k].cpu().numpy(), outs[0][1][k].cpu().numpy(), rtol=2e-5)


def test_empty_layer_decodes_to_zero():
    w = WORKLOADS["tiny"]
    gpu, _ = make_pair(w)
    out, m = gpu.decode(0, to_dev(gen_q(w, 0, 0), w), w.delta_req)
    assert torch.count_nonzero(out) == 0
    assert torch.count_nonzero(m["meter_a"]) == 0 and torch.count_nonzero(m["meter_b"]) == 0


@pytest.mark.parametrize("scheme,v_witness,batch,pages", [
    ("fp8_e4m3", False, 2, 0), ("blackbox", True, 2, 0), ("int8_dither", False, 2, 0), ("int8_dither", True, 2, 0),
    ("int8_dither", True, 1, 0),         # one sequence: single-warp CTAs, key dither in registers
    ("int8_dither", False, 1, 40),       # the same, paged
])
def test_gate_decisions_bit_exact_and_repaired_decode(scheme, v_witness, batch, pages):
    """Raw-cast FP8, the black-box store and dithered INT8 (ranked by its Tier B risks): the GPU's
    block risks match the oracle's (never below, within 1e-4); the oracle's gate, fed the GPU's
    block risks, picks exactly the blocks the GPU pages in, and fed its own risks picks them too
    outside the tie zone (empty here); the next decode matches the oracle on the repaired cache
    (value witnesses stay: the gate pages in keys only)."""
    w = WORKLOADS["qwen_1l"].with_(batch=batch, context=400, steps=3, scheme=scheme)
    gpu, ref = make_pair(w, gate_blocks=2 * 4 * 32, v_witness=v_witness, max_pages=pages)
    K, V = gen_kv(w, 0)
    write_both(gpu, ref, 0, K, V, w)
    taus = (0.5, 0.2, 0.05) if scheme != "int8_dither" else (4.0, 2.0, 1.0)
    for step, tau in enumerate(taus):
        q = gen_q(w, 0, step)
        _, _, r = check_decode(gpu, ref, 0, q, w, w.delta_req)
        risk = gpu.export(0, _lib.X_BLOCK_RISK).cpu().numpy()
        check_risk(risk, r["risk"], what=f"block risk step {step}")
        before = ref.repaired[0].copy()
        gpu.witcert_gate(0, tau)
        picked = ref.gate(0, tau, risk)
        slots = gpu.export(0, _lib.X_SLOTS).cpu().numpy()
        np.testing.assert_array_equal(slots >= 0, ref.repaired[0])
        assert len(picked) == len(set(picked))
        assert check_gate_end_to_end(r["risk"], before, tau, slots >= 0, w.group) == 0
    check_decode(gpu, ref, 0, gen_q(w, 0, 9), w, w.delta_req)
    st = gpu.witcert_gate_stats()
    assert st["blocks_paged_in"] == int(ref.repaired[0].sum()) > 0
    assert st["bytes_paged_in"] == st["blocks_paged_in"] * 16 * 128 * 2
    # appends into a repaired partial block keep the exact pool row in step
    k1, v1 = gen_append_kv(w, 0, 0)
    write_both(gpu, ref, 0, k1, v1, w, seed=3)
    check_decode(gpu, ref, 0, gen_q(w, 0, 10), w, w.delta_req)


@pytest.mark.parametrize("delta_req,n_splits", [(1e-2, 8), (1e-3, 0)])
def test_full_28_layer_config_sampled_cells(delta_req, n_splits):
    """Full-size Qwen decode shape (B=16 x 4096, 28q/4kv), two of its 28 layers written and
    decoded with the configured 8 KV splits and with the automatic split count the bench
    uses; sampled (seq, KV head) groups are checked against the oracle computed for those
    groups alone."""
    w = WORKLOADS["qwen_28l"].with_(n_layers=28, steps=64)
    gpu, _ = make_pair(w, n_splits=n_splits, extra_tokens=1)
    dl = meter.delta_loc(delta_req, w.n_layers, w.n_q_heads, w.steps)
    for layer in (0, 27):
        K, V = gen_kv(w, layer)
        gpu.witcert_write(layer, to_dev(K, w), to_dev(V, w))
        q = gen_q(w, layer, 0)
        out, m = gpu.decode(layer, to_dev(q, w), delta_req)
        o = out.cpu().numpy()
        for i, h in [(0, 0), (7, 3), (15, 1)]:
            js = slice(h * w.group, (h + 1) * w.group)
            r = oracle_group(w, layer, K[i, :, h], V[i, :, h], q[i, js], i, h, w.scheme, dl)
            assert np.abs(o[i, js] - r["out"]).max() <= 2e-3 * np.abs(V[i, :, h]).max()
            check_meter(m["raw_a"].cpu().numpy()[i, js], r["raw_a"], what="raw_a", raw=True)
            check_meter(m["raw_b"].cpu().numpy()[i, js], r["raw_b"], what="raw_b", raw=True)


def test_errors_are_reported_not_raised_on_device():
    w = WORKLOADS["tiny"]
    gpu, _ = make_pair(w)
    K, V = gen_kv(w, 0)
    with pytest.raises(wc.WitcertError) as e:
        big = np.concatenate([K] * 2, 1)
        gpu.witcert_write(0, to_dev(big, w), to_dev(big, w))
    assert e.value.status == _lib.EINVAL and "capacity" in str(e.value)
    gpu.witcert_write(0, to_dev(K, w), to_dev(V, w))
    with pytest.raises(wc.WitcertError) as e:
        gpu.decode(0, to_dev(gen_q(w, 0, 0), w), 0.0)
    assert e.value.status == _lib.EINVAL
    with pytest.raises(wc.WitcertError) as e:
        gpu.witcert_gate(0, 1.0)
    assert e.value.status == _lib.ESTATE
    assert gpu.witcert_stats()["device_errors"] == 0


@pytest.mark.parametrize("scheme", ALL_SCHEMES)
def test_witness_fallback_on_extreme_keys(scheme):
    """Keys near 1e-20 and near 1e25 push the writers' fp32 double-float witness outside its
    safe range, so those bands take the fp64 computation; keys near 1e-9 give witnesses in
    fp16's subnormal range.  Values scaled the same way do this to the value witnesses.  Every
    stored witness must still equal the oracle's bit for bit."""
    w = WORKLOADS["tiny"].with_(scheme=scheme)
    K, V = gen_kv(w, 0)
    K = K.copy()
    K[:, 0:5] *= 1e-20         # residuals far below 2^-45
    K[:, 5:9] *= 1e25          # residuals above 2^60
    K[:, 9:13] *= 1e-9         # witnesses below fp16's smallest normal
    V = V.copy()               # the same for the value witnesses
    V[:, 0:5] *= 1e-20
    V[:, 5:9] *= 1e25
    V[:, 9:13] *= 1e-9
    gpu, ref = make_pair(w, v_witness=True)
    write_both(gpu, ref, 0, K, V, w)
    check_write(gpu, ref, 0, scheme)
