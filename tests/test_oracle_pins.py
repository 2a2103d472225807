"""The float64 oracle against values fixed by the pages and by mathematics."""
import pytest

from oracle import moe_oracle as O
from tests.oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(O)
