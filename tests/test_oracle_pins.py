"""The fp64 oracle against hand-derived values, library routines and exact
algebraic properties (no GPU)."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()
