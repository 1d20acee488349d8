"""The fp64 oracle against exact brute force, closed forms and library routines (CPU)."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(O, pin):
    pin(O)
