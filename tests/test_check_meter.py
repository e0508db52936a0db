"""The meter comparison the GPU parity tests use accepts only values that bound the oracle's
from above within the relative tolerance (CPU only)."""
import numpy as np
import pytest

from gpu_helpers import METER_REL, check_meter


def test_accepts_equal_and_slightly_above():
    r = np.array([0.0, 1e-6, 0.25, np.inf])
    check_meter(r, r)
    check_meter(r * (1 + METER_REL / 2), r)


@pytest.mark.parametrize("bad", [
    np.array([0.25 * (1 - 1e-5)]),        # below the oracle: not a bound
    np.array([np.nextafter(0.25, 0.0)]),  # one unit below is below too: no relative slack
    np.array([0.25 * (1 + 1e-3)]),        # looser than the tolerance
    np.array([np.nan]),                   # a NaN fails both comparisons and bounds nothing
])
def test_rejects_below_above_and_nan(bad):
    with pytest.raises(AssertionError):
        check_meter(bad, np.array([0.25]))


def test_absolute_allowance_is_for_values_below_fp32_range_only():
    check_meter(np.array([0.0]), np.array([3.5e-90]))            # a value no fp32 meter can carry
    with pytest.raises(AssertionError):
        check_meter(np.array([0.0]), np.array([1e-20]))


def test_raw_meters_above_one_are_held_to_the_tolerance_on_d():
    # D = 9023.25: raw = D + D^2/2; D 6e-5 above passes (raw then 1.2e-4 above), 2e-4 above does not
    d = 9023.25
    raw = lambda x: x + x * x / 2
    check_meter(np.array([raw(d * (1 + 6e-5))]), np.array([raw(d)]), raw=True)
    with pytest.raises(AssertionError):
        check_meter(np.array([raw(d * (1 + 6e-5))]), np.array([raw(d)]))
    with pytest.raises(AssertionError):
        check_meter(np.array([raw(d * (1 + 2e-4))]), np.array([raw(d)]), raw=True)
    with pytest.raises(AssertionError):                           # below stays below
        check_meter(np.array([np.nextafter(raw(d), 0.0)]), np.array([raw(d)]), raw=True)
    # at or below 1 the raw value is the meter: the tolerance stays on it
    with pytest.raises(AssertionError):
        check_meter(np.array([0.9 * (1 + 1.5e-4)]), np.array([0.9]), raw=True)
