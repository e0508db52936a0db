"""witcert_decode_noalloc: the metered decode for callers that cannot allocate device memory.

Serving engines that give all free device memory to their own pool or caching
allocator at start-up, and hosts that forbid device allocation after start-up,
cannot let a library call cudaMalloc on their decode path.  This entry point
keeps its split scratch in a static device array instead.  These tests call it
through the C ABI and compare it with witcert_decode on the same cache, on two
calls in a row (the second reuses the array the first call left behind).  Both
run the same kernels with the same split count, so every output, meter and
block risk must be bit-identical.  The file is named to run last, so a failure
here never hides another test.
"""
import numpy as np
import pytest
import torch

import kv_cache_quantization_witcert_gb300 as wc
from kv_cache_quantization_witcert_gb300 import _lib
from workload import WORKLOADS, gen_kv, gen_q

from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu

NAMES = ("meter_a", "meter_b", "raw_a", "raw_b", "meter_v")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    wc.load()


def both_decodes(cache, q, delta_req, v_witness):
    """(out, meters) of witcert_decode, then of witcert_decode_noalloc into NaN-filled buffers."""
    res = []
    for call in (cache.witcert_decode, cache.witcert_decode_noalloc):
        B, Hq = q.shape[0], q.shape[1]
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        m = torch.full((5, B, Hq), float("nan"), dtype=torch.float32, device="cuda")
        call(0, q, delta_req, out, m[0], m[1], m[2], m[3], m[4] if v_witness else None)
        torch.cuda.synchronize()
        res.append((out, m))
    return res


@pytest.mark.parametrize("scheme", ["int8_dither", "fp8_e4m3"])
def test_noalloc_decode_is_bit_identical_on_two_calls(scheme):
    w = WORKLOADS["qwen_1l"].with_(batch=5, context=1500, scheme=scheme)
    cache = wc.Cache(w.n_layers, w.n_q_heads, w.n_kv_heads, w.batch, w.context, scheme,
                     dtype=torch.bfloat16, seed=w.seed, total_steps=w.steps)
    K, V = gen_kv(w, 0)
    cache.witcert_write(0, to_dev(K, w), to_dev(V, w))
    calls0 = cache.witcert_stats()["decode_calls"]
    for step in (0, 1):
        (o1, m1), (o2, m2) = both_decodes(cache, to_dev(gen_q(w, 0, step), w), w.delta_req, False)
        assert torch.isfinite(o2).all()
        assert torch.equal(o1, o2), f"out, call {step}"
        assert torch.equal(m1[:4], m2[:4]) or (scheme != "int8_dither" and torch.equal(m1[[0, 2]], m2[[0, 2]])), step
    st = cache.witcert_stats()
    assert st["decode_calls"] == calls0 + 4 and st["last_n_splits"] > 0
    cache.close()


TEN = [600, 75, 333, 0, 1, 599, 16, 17, 300, 450]


@pytest.mark.parametrize("scheme,lens", [("int8_dither", [600, 75, 333]), ("int8_dither", TEN), ("fp8_e4m3", TEN)])
def test_noalloc_keeps_the_gate_risks_and_ragged_value_meter(scheme, lens):
    """A gated, ragged cache with value witnesses: the block risks the gate reads and the value
    meter are the same bits through either entry point, and the gate after a no-allocation
    decode pages in the same blocks.  Three sequences (split CTAs of 2 warps), ten (8 warps), and
    ten of the raw-cast FP8 scheme (one warp per sequence and block range)."""
    w = WORKLOADS["qwen_1l"].with_(batch=len(lens), context=600, scheme=scheme)
    runs = []
    for noalloc in (False, True):
        cache = wc.Cache(1, w.n_q_heads, w.n_kv_heads, w.batch, 640, scheme, dtype=torch.bfloat16,
                         seed=w.seed, total_steps=w.steps, max_repair_blocks=w.batch * 4 * 40, v_witness=True)
        K, V = gen_kv(w, 0)
        Kp = np.concatenate([K[i, :n] for i, n in enumerate(lens)])
        Vp = np.concatenate([V[i, :n] for i, n in enumerate(lens)])
        cache.witcert_write_ragged(0, to_dev(Kp, w), to_dev(Vp, w), lens)
        for step in (0, 1):
            q = to_dev(gen_q(w, 0, step), w)
            out = torch.empty((w.batch, w.n_q_heads, 128), dtype=torch.float32, device="cuda")
            m = torch.empty((5, w.batch, w.n_q_heads), dtype=torch.float32, device="cuda")
            call = cache.witcert_decode_noalloc if noalloc else cache.witcert_decode
            call(0, q, w.delta_req, out, m[0], m[1], m[2], m[3], m[4])
            risk = cache.export(0, _lib.X_BLOCK_RISK)
            cache.witcert_gate(0, 4.0 if scheme == "int8_dither" else 0.5)
            slots = cache.export(0, _lib.X_SLOTS)
            torch.cuda.synchronize()
            runs.append((out.clone(), m.clone(), risk.clone(), slots.clone()))
        cache.close()
    n = len(runs) // 2
    for k in range(n):
        (o1, m1, r1, s1), (o2, m2, r2, s2) = runs[k], runs[n + k]
        assert torch.equal(o1, o2), f"step {k}"
        # the same bits, NaN where the scheme has no Tier B (FP8: meter_b and raw_b)
        torch.testing.assert_close(m1, m2, rtol=0, atol=0, equal_nan=True, msg=f"meters, step {k}")
        assert torch.equal(r1, r2), f"block risks, step {k}"
        assert torch.equal(s1 >= 0, s2 >= 0), f"repaired blocks, step {k}"
    assert (runs[-1][3] >= 0).any()


def test_noalloc_rejects_shapes_beyond_the_static_array():
    # 64 sequences x 32 query heads x 64 splits x 544 bytes = 71 MB > 16 MiB
    cache = wc.Cache(1, 32, 4, 64, 64, "fp8_e4m3", dtype=torch.bfloat16, n_splits=64)
    q = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((64, 32, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(wc.WitcertError) as e:
        cache.witcert_decode_noalloc(0, q, 1e-2, out)
    assert e.value.status == _lib.EINVAL and "static" in str(e.value)
    cache.close()
