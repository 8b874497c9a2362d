"""The fp64 oracle against closed forms, invariants, finite differences,
a hand-worked example and PyTorch's fp64 CPU attention (CPU only)."""
import pytest

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin()
