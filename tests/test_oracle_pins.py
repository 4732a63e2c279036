"""The CPU oracle against its pins (brute force, library routines, closed
forms, the identities the pages fix, the degree-rule table)."""
import pytest

import oracle
from pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle.tp_oracle)
