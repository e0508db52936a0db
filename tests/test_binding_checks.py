"""The Python binding rejects tensors of the wrong device, dtype, shape or layout before any
library call (CPU only: the checks run before the C ABI is reached, so no cache is created)."""
import pytest
import torch

import kv_cache_quantization_witcert_gb300 as wc
from kv_cache_quantization_witcert_gb300 import _lib

B, HQ, HKV = 2, 8, 2


@pytest.fixture
def cache():
    c = object.__new__(wc.Cache)          # no witcert_create: every call below must fail first
    c.cfg = _lib.witcert_config(1, HQ, HKV, 128, B, 64, 0, _lib.BF16, 0, 1, 0, 0, 0, 0, 0)
    c.dtype = torch.bfloat16
    c.v_witness = False
    c._h = None
    return c


def kv(n=3, dtype=torch.bfloat16):
    return torch.zeros((B, n, HKV, 128), dtype=dtype)


def test_write_rejects_host_tensors_and_mismatches(cache):
    with pytest.raises(ValueError, match="CUDA"):
        cache.witcert_write(0, kv(), kv())
    with pytest.raises(ValueError, match="dtype|bfloat16"):
        cache.witcert_write(0, kv(dtype=torch.float32), kv())
    with pytest.raises(ValueError, match="shape"):
        cache.witcert_write(0, kv(3), kv(4))                       # V holds another token count
    with pytest.raises(ValueError, match="shape"):
        cache.witcert_write(0, torch.zeros((B, HKV, 3, 128), dtype=torch.bfloat16), kv())
    with pytest.raises(ValueError, match="contiguous"):
        cache.witcert_write(0, kv().transpose(1, 2), kv())
    with pytest.raises(ValueError, match="None"):
        cache.witcert_write_hat(0, kv(), kv(), None, kv())


def test_ragged_write_checks_counts_and_packed_rows(cache):
    packed = torch.zeros((5, HKV, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="per sequence"):
        cache.witcert_write_ragged(0, packed, packed, [5])
    with pytest.raises(ValueError, match="shape"):
        cache.witcert_write_ragged(0, packed, packed, [2, 2])      # 4 rows counted, 5 given
    with pytest.raises(ValueError, match="CUDA"):
        cache.witcert_write_ragged(0, packed, packed, [2, 3])


def test_decode_checks_every_output_buffer(cache):
    q = torch.zeros((B, HQ, 128), dtype=torch.bfloat16)
    out = torch.zeros((B, HQ, 128), dtype=torch.float32)
    with pytest.raises(ValueError, match="out"):
        cache.witcert_decode(0, q, 1e-2, torch.zeros((B, HQ, 64), dtype=torch.float32))
    with pytest.raises(ValueError, match="meter_a"):
        cache.witcert_decode(0, q, 1e-2, out, torch.zeros((B, HQ - 1), dtype=torch.float32))
    with pytest.raises(ValueError, match="meter_v"):
        cache.witcert_decode_noalloc(0, q, 1e-2, out, meter_v=torch.zeros((B, HQ), dtype=torch.float16))
    with pytest.raises(ValueError, match="part"):
        cache.witcert_decode_partial(0, q, 1e-2, 64, torch.zeros((B, HQ, 128), dtype=torch.float32))
    with pytest.raises(ValueError, match="CUDA"):
        cache.witcert_decode(0, q, 1e-2, out)


def test_merge_and_export_reject_host_buffers(cache):
    parts = torch.zeros((B, HQ, 2, wc.PART_STRIDE), dtype=torch.float32)
    with pytest.raises(ValueError, match="parts"):
        wc.witcert_merge_partials(parts[..., :100].contiguous(), "int8_dither")
    with pytest.raises(ValueError, match="CUDA"):
        wc.witcert_merge_partials(parts, "int8_dither", out=torch.zeros((B, HQ, 128), dtype=torch.float32))
    with pytest.raises(ValueError, match="CUDA"):
        cache.witcert_export(0, _lib.X_WITNESS, torch.zeros(16, dtype=torch.float16))


def test_non_tensor_arguments_are_named(cache):
    import numpy as np
    with pytest.raises(ValueError, match="K must be a torch.Tensor"):
        cache.witcert_write(0, np.zeros((B, 3, HKV, 128), np.float32), kv())
    with pytest.raises(ValueError, match="q must be a torch.Tensor"):
        cache.witcert_decode(0, [[0.0]], 1e-2, torch.zeros((B, HQ, 128), dtype=torch.float32))
