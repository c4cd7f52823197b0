"""The oracle against its pins (library routines, closed forms, invariants, page examples)."""
import pytest

import oracle_pins
from oracle import oracle as O


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(O.default())
