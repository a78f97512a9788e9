"""The oracle against its pins (see ``oracle_pins.py`` for what pins what)."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.load())
