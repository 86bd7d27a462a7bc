"""The fp64 oracle against its pins (CPU only)."""
import pytest

import oracle
from tests.oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.default())
