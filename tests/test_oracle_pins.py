"""The fp64 oracle against its pins: closed forms, hand-derived golden values,
library routines on special cases, and the invariants the pages state."""
import pytest

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(oracle, pin):
    pin(oracle)
