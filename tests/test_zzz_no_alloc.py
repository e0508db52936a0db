"""witcert_decode_noalloc: the metered decode for callers that cannot allocate device memory.

Serving engines that give all free device memory to their own pool or caching
allocator at start-up, and hosts that forbid device allocation after start-up,
cannot let a library call cudaMalloc on their decode path.  This entry point
keeps its split scratch in a static device array instead.  These tests call it
through the C ABI and compare it with witcert_decode on the same cache, on two
calls in a row (the second reuses the array the first call left behind).
The file is named to run last, so a failure here never hides another test.
"""
import numpy as np
import pytest
import torch

import kv_cache_quantization_witcert_gb300 as wc
from kv_cache_quantization_witcert_gb300 import _lib
from workload import WORKLOADS, gen_kv, gen_q

from gpu_helpers import METER_REL, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    wc.load()


@pytest.mark.parametrize("scheme", ["int8_dither", "fp8_e4m3"])
def test_noalloc_decode_matches_decode_on_two_calls(scheme):
    w = WORKLOADS["qwen_1l"].with_(batch=5, context=1500, scheme=scheme)
    cache = wc.Cache(w.n_layers, w.n_q_heads, w.n_kv_heads, w.batch, w.context, scheme,
                     dtype=torch.bfloat16, seed=w.seed, total_steps=w.steps)
    K, V = gen_kv(w, 0)
    cache.witcert_write(0, to_dev(K, w), to_dev(V, w))
    vmax = float(np.abs(V).max())
    for call, step in enumerate((0, 1)):
        q = to_dev(gen_q(w, 0, step), w)
        ref_out, ref_m = cache.decode(0, q, w.delta_req)
        out = torch.full_like(ref_out, float("nan"))
        m = torch.full((4, w.batch, w.n_q_heads), float("nan"), dtype=torch.float32, device="cuda")
        cache.witcert_decode_noalloc(0, q, w.delta_req, out, m[0], m[1], m[2], m[3])
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert (out - ref_out).abs().max().item() <= 2e-3 * vmax, f"call {call}"
        for k, idx in (("meter_a", 0), ("raw_a", 2)) + ((("meter_b", 1), ("raw_b", 3)) if scheme == "int8_dither" else ()):
            g = m[idx].cpu().numpy().astype(np.float64)
            r = ref_m[k].cpu().numpy().astype(np.float64)
            np.testing.assert_allclose(g, r, rtol=METER_REL, atol=0, err_msg=f"{k} call {call}")
    cache.close()


def test_noalloc_rejects_shapes_beyond_the_static_array():
    # 64 sequences x 32 query heads x 64 splits x 544 bytes = 71 MB > 16 MiB
    cache = wc.Cache(1, 32, 4, 64, 64, "fp8_e4m3", dtype=torch.bfloat16, n_splits=64)
    q = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((64, 32, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(wc.WitcertError) as e:
        cache.witcert_decode_noalloc(0, q, 1e-2, out)
    assert e.value.status == _lib.EINVAL and "static" in str(e.value)
    cache.close()
