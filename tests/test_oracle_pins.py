"""The float64 oracle against its pins (closed forms, library routines, brute force, page values)."""
import pytest

import oracle_pins
from oracle import dflash_oracle as O


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(O)
