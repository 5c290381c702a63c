"""The CPU oracle against the pages' worked examples, library routines, brute force and invariants."""
import pytest

from oracle import quoka_oracle
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(quoka_oracle)
