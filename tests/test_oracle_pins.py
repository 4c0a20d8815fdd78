"""The CPU oracle against the pages' worked examples, closed forms, invariants and the independent
1-semiseparable / convolution evaluations (see oracle_pins.py for each pin's source)."""
import pytest

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(orc, pin):
    pin(orc)
