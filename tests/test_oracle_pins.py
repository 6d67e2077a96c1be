"""The CPU oracle against the pins (closed forms, invariants, brute force, golden values)."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(oracle_impl, pin):
    pin(oracle_impl)
