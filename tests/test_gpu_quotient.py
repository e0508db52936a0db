"""The INT8 writer's quotient x / s against the IEEE quotient (needs a GB300).

The writer divides each element by its group's fp16 scale with a correctly rounded reciprocal
and one exact correction (Markstein's theorem).  The self test compares that with the IEEE
quotient for every positive fp16 scale, against every bfloat16 x the writer can meet with that
scale and seeded float32 x, wherever the quotient can move a code; the codes themselves are
checked bit for bit against the oracle by the parity tests.
"""
import pytest
import torch

import kv_cache_quantization_witcert_gb300 as wc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    wc.load()


@pytest.mark.parametrize("seed", [0, 12345])
def test_quotient_equals_ieee_division_for_every_fp16_scale(seed):
    assert wc.witcert_quotient_selftest(n_f32=8192, seed=seed) == 0
