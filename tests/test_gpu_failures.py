"""Failure paths on the GPU, none of which faults, traps or hangs the device.

* The bounded shared-memory barrier wait of the decode pipeline gives up after its
  limit when nothing completes the barrier, reports a timeout, and the context
  stays usable.
* The gate with an exact-key pool too small for what it selects pages in what fits,
  counts the rest as dropped, leaves the dropped blocks' witnesses in place, and the
  meters of the next decode stay sound (they match the oracle on the blocks actually
  repaired).
"""
import numpy as np
import pytest
import torch

import kv_cache_quantization_witcert_gb300 as wc
from kv_cache_quantization_witcert_gb300 import _lib
from workload import WORKLOADS, gen_kv, gen_q

from gpu_helpers import check_decode, make_pair, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    wc.load()


def test_bounded_device_wait_times_out_and_context_survives():
    assert wc.witcert_wait_selftest(2_000_000) == _lib.ETIMEDOUT          # 2 ms, nothing arrives
    assert b"gave up" in _lib.load().witcert_last_error()
    w = WORKLOADS["tiny"]
    gpu, ref = make_pair(w)
    K, V = gen_kv(w, 0)
    gpu.witcert_write(0, to_dev(K, w), to_dev(V, w))
    ref.write(0, K, V)
    check_decode(gpu, ref, 0, gen_q(w, 0, 0), w, w.delta_req)


def test_gate_with_exhausted_pool_drops_and_stays_sound():
    w = WORKLOADS["qwen_1l"].with_(batch=2, context=400, steps=3, scheme="fp8_e4m3")
    cap = 3
    gpu, ref = make_pair(w, gate_blocks=cap)
    K, V = gen_kv(w, 0)
    gpu.witcert_write(0, to_dev(K, w), to_dev(V, w))
    ref.write(0, K, V)
    check_decode(gpu, ref, 0, gen_q(w, 0, 0), w, w.delta_req)
    risk = gpu.export(0, _lib.X_BLOCK_RISK).cpu().numpy()
    gpu.witcert_gate(0, 0.05)
    wanted = set(ref.gate(0, 0.05, risk))
    assert len(wanted) > cap
    slots = gpu.export(0, _lib.X_SLOTS).cpu().numpy()
    got = {(i, h, b) for i, h, b in zip(*np.nonzero(slots >= 0))}
    assert len(got) == cap and got <= wanted
    st = gpu.witcert_gate_stats()
    assert st["blocks_paged_in"] == cap and st["blocks_dropped"] == len(wanted) - cap
    wit = gpu.export(0, _lib.X_WITNESS).cpu().numpy()
    for i, h, b in wanted - got:                     # dropped: witnesses untouched
        assert np.any(wit[i, 16 * b:16 * b + 16, h] > 0)
    for i, h, b in got:                              # repaired: witnesses zeroed
        assert np.all(wit[i, 16 * b:16 * b + 16, h] == 0)
    ref.repaired[0][:] = slots >= 0                  # the oracle on what was really repaired
    check_decode(gpu, ref, 0, gen_q(w, 0, 1), w, w.delta_req)


def test_lost_backing_store_fails_the_gate_and_changes_nothing():
    """A page-in that cannot complete (the layer's backing store lost its exact keys, injected on
    the host as a failed copy would leave it): the gate returns EPAGEIN, selects, pages in and
    zeroes nothing, and the next decode's meters still bound the oracle's on the unrepaired
    cache; another layer's gate still works."""
    w = WORKLOADS["qwen_1l"].with_(n_layers=2, batch=2, context=400, steps=3, scheme="fp8_e4m3")
    gpu, ref = make_pair(w, gate_blocks=2 * 4 * 32)
    for layer in (0, 1):
        K, V = gen_kv(w, layer)
        gpu.witcert_write(layer, to_dev(K, w), to_dev(V, w))
        ref.write(layer, K, V)
        check_decode(gpu, ref, layer, gen_q(w, layer, 0), w, w.delta_req)
    wit0 = gpu.export(0, _lib.X_WITNESS).cpu().numpy()
    gpu.witcert_inject_fault(_lib.FAULT_BACKING_LOST, 0)
    with pytest.raises(wc.WitcertError) as e:
        gpu.witcert_gate(0, 0.05)
    assert e.value.status == _lib.EPAGEIN
    assert np.all(gpu.export(0, _lib.X_SLOTS).cpu().numpy() < 0)
    np.testing.assert_array_equal(gpu.export(0, _lib.X_WITNESS).cpu().numpy().view(np.uint16), wit0.view(np.uint16))
    st = gpu.witcert_gate_stats()
    assert st["blocks_paged_in"] == 0 and st["cells_triggered"] == 0
    check_decode(gpu, ref, 0, gen_q(w, 0, 1), w, w.delta_req)      # unrepaired oracle: nothing moved
    gpu.witcert_gate(1, 0.05)                                        # layer 1 keeps its backing store
    assert gpu.witcert_gate_stats()["blocks_paged_in"] > 0
    with pytest.raises(wc.WitcertError) as e:                        # the fault persists
        gpu.witcert_gate(0, 0.05)
    assert e.value.status == _lib.EPAGEIN
    assert gpu.witcert_stats()["device_errors"] == 0
