"""The meter comparison the GPU parity tests use accepts only values that bound the oracle's
from above within the relative tolerance (CPU only)."""
import numpy as np
import pytest

from gpu_helpers import FP32_ULP, METER_REL, check_meter


def test_accepts_equal_and_slightly_above():
    r = np.array([0.0, 1e-6, 0.25, np.inf])
    check_meter(r, r)
    check_meter(r * (1 + METER_REL / 2), r)
    check_meter(r * (1 - FP32_ULP / 2), r)


@pytest.mark.parametrize("bad", [
    np.array([0.25 * (1 - 1e-5)]),        # below the oracle: not a bound
    np.array([0.25 * (1 + 1e-3)]),        # looser than the tolerance
    np.array([np.nan]),                   # a NaN fails both comparisons and bounds nothing
])
def test_rejects_below_above_and_nan(bad):
    with pytest.raises(AssertionError):
        check_meter(bad, np.array([0.25]))
