"""Degenerate inputs of the quantizers and the meter, on the GPU against the oracle.

All-zero tokens give every INT8 group amax 0 (scale 0, codes 0) and every KIVI block and
group max = min (scale 0); a zero 32-channel group sits inside an otherwise normal token;
one 16-token block has keys constant over the block in every channel (KIVI's per-channel
scale is 0 and the zero point carries the value); one value group is constant; one query
head is all zero (Tier A and Tier B terms are exactly 0, so both meters are 0 and the
output is the plain mean of the values).
"""
import numpy as np
import pytest
import torch

import kv_cache_quantization_witcert_gb300 as wc
from workload import WORKLOADS, gen_kv, gen_q

from gpu_helpers import check_decode, check_write, make_pair, write_both

pytestmark = pytest.mark.gpu

ALL_SCHEMES = ["int8_dither", "fp8_e4m3", "kivi2", "int8_rtn", "blackbox"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    wc.load()


@pytest.mark.parametrize("base", ["tiny", "qwen_1l"])
@pytest.mark.parametrize("scheme", ALL_SCHEMES)
def test_zero_and_constant_inputs(scheme, base):
    w = WORKLOADS[base].with_(batch=2, context=64, steps=2, scheme=scheme)
    gpu, ref = make_pair(w, v_witness=True)
    K, V = gen_kv(w, 0)
    K, V = K.copy(), V.copy()
    K[:, 0:16] = 0.0                      # block 0: all-zero tokens
    V[:, 0:16] = 0.0
    K[:, 20, :, 32:64] = 0.0              # one zero group inside token 20
    V[:, 20, :, 32:64] = 0.0
    K[:, 32:48] = K[:, 32:33]             # block 2: every channel constant over the block
    V[:, 40, :, 64:96] = 0.75             # one constant value group
    write_both(gpu, ref, 0, K, V, w)
    check_write(gpu, ref, 0, scheme)
    q = gen_q(w, 0, 0).copy()
    q[:, 0] = 0.0                         # query head 0 of every sequence
    _, m, r = check_decode(gpu, ref, 0, q, w, w.delta_req)
    assert np.all(m["raw_a"].cpu().numpy()[:, 0] == 0.0) and np.all(r["raw_a"][:, 0] == 0.0)
    assert gpu.witcert_stats()["device_errors"] == 0
