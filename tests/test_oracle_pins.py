"""CPU pins of the fp64 oracle (no GPU): see ``oracle_pins`` for the sources."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle)
