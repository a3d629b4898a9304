"""CPU pins of the fp64 oracle (no GPU): see ``oracle_pins`` for the sources."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle)


from oracle_pins import BACKWARD_PINS  # noqa: E402
import oracle.attention as fwd_mod  # noqa: E402
import oracle.attention_grad as bwd_mod  # noqa: E402


@pytest.mark.parametrize("pin", BACKWARD_PINS, ids=lambda f: f.__name__)
def test_backward_pin(pin):
    pin(fwd_mod, bwd_mod)
