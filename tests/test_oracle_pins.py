"""The fp64 oracle against the pages' printed values, closed forms, invariants,
library routines it does not call, and brute force (CPU only)."""
import pytest

import oracle_pins

PINS = oracle_pins.ALL_PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()
