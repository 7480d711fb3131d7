"""The CPU oracle against the pages' printed values, closed forms, library
routines, brute force and invariants (no GPU needed)."""
import pytest

import oracle
from tests import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle)
