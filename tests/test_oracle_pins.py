"""The oracle against its pins (no GPU): worked examples, closed forms, invariants."""
import pytest

from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(orc, pin):
    pin(orc)
