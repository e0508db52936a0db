"""Context-parallel decode on one GPU: shards of one context in separate caches.

Two caches hold positions [0, 512) and [512, 1000) of every sequence (the second
created with pos_offset=512, so its dither is keyed on global positions); each
decodes its slice with witcert_decode_partial and witcert_merge_partials merges
the two shards' records.  The result must match the oracle decoding the whole
context in one piece, within the same tolerances as a single-cache decode; the
value meter rides in the records too.
"""
import numpy as np
import pytest
import torch

import kv_cache_quantization_witcert_gb300 as wc
from kv_cache_quantization_witcert_gb300 import _lib
from workload import WORKLOADS, gen_kv, gen_q

from gpu_helpers import METER_REL, check_meter, make_pair, to_dev, torch_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    wc.load()


def _shard(w, scheme, K, V, lo, hi):
    c = wc.Cache(w.n_layers, w.n_q_heads, w.n_kv_heads, w.batch, hi - lo, scheme, dtype=torch_dtype(w),
                 seed=w.seed, total_steps=w.steps, pos_offset=lo, v_witness=True)
    c.witcert_write(0, to_dev(K[:, lo:hi], w), to_dev(V[:, lo:hi], w))
    return c


@pytest.mark.parametrize("scheme", ["int8_dither", "fp8_e4m3"])
def test_two_shards_merge_to_the_whole_context(scheme):
    w = WORKLOADS["qwen_1l"].with_(batch=3, context=1000, steps=1, scheme=scheme)
    K, V = gen_kv(w, 0)
    _, ref = make_pair(w, v_witness=True)
    ref.write(0, K, V)
    shards = [_shard(w, scheme, K, V, 0, 512), _shard(w, scheme, K, V, 512, 1000)]
    # the shards' stores are the whole cache's, slice by slice
    full = wc.Cache(w.n_layers, w.n_q_heads, w.n_kv_heads, w.batch, 1000, scheme, dtype=torch_dtype(w),
                    seed=w.seed, total_steps=w.steps, v_witness=True)
    full.witcert_write(0, to_dev(K, w), to_dev(V, w))
    for kind in (_lib.X_K_CODES, _lib.X_V_CODES, _lib.X_WITNESS, _lib.X_V_WITNESS):
        whole = full.export(0, kind).cpu()
        parts = torch.cat([s.export(0, kind).cpu() for s in shards], dim=1)
        assert torch.equal(whole, parts)
    q = to_dev(gen_q(w, 0, 0), w)
    recs = torch.stack([s.decode_partial(0, q, w.delta_req, 1000) for s in shards], dim=2).contiguous()
    out, m = wc.witcert_merge_partials(recs, scheme)
    torch.cuda.synchronize()
    ref.w16[0] = full.export(0, _lib.X_WITNESS).cpu().numpy()
    ref.wv16[0] = full.export(0, _lib.X_V_WITNESS).cpu().numpy()
    r = ref.decode(0, gen_q(w, 0, 0), w.delta_req)
    vmax = float(np.abs(V).max())
    assert np.abs(out.cpu().numpy() - r["out"]).max() <= 2e-3 * vmax
    check_meter(m["raw_a"].cpu().numpy(), r["raw_a"], METER_REL, "raw_a", raw=True)
    check_meter(m["meter_v"].cpu().numpy(), r["meter_v"], METER_REL, "meter_v")
    if scheme == "int8_dither":
        check_meter(m["raw_b"].cpu().numpy(), r["raw_b"], METER_REL, "raw_b", raw=True)
    for c in shards + [full]:
        assert c.witcert_stats()["device_errors"] == 0
        c.close()


def test_partial_decode_rejects_a_total_shorter_than_its_slice():
    w = WORKLOADS["qwen_1l"].with_(batch=2, context=64, steps=1, scheme="fp8_e4m3")
    K, V = gen_kv(w, 0)
    c = _shard(w, "fp8_e4m3", K, V, 0, 64)
    q = to_dev(gen_q(w, 0, 0), w)
    with pytest.raises(wc.WitcertError) as e:
        c.decode_partial(0, q, w.delta_req, 32)
    assert e.value.status == _lib.EINVAL
    c.close()
