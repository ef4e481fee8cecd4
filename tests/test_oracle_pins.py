"""The fp64 oracle against its pins (brute force, library routine, closed forms, invariants)."""

import pytest

import oracle
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle)
