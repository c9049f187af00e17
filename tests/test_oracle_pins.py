"""The fp64 oracle against what the pages and mathematics fix (no GPU)."""
import pytest

import oracle
from pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle.default)
