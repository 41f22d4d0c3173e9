"""The CPU oracle against what the pages and mathematics fix (see oracle_pins)."""
import pytest

import oracle_pins
from oracle import irs_oracle


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(irs_oracle)
