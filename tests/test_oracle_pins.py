"""The oracle against facts it does not produce itself (see ``oracle_pins.py``)."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__[4:])
def test_pin(pin):
    pin(oracle.lib())
