"""The CPU oracle against its pins (no GPU). See ``oracle_pins.py``."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin()
