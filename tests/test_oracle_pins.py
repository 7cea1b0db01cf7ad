"""The oracle against its pins (tests/oracle_pins.py); CPU only."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda f: f.__name__[6:])
def test_pin(check):
    check(oracle.default())
