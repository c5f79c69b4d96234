"""The oracle against its pins (CPU only).  See tests/oracle_pins.py for what
each pin checks and which page section fixes it."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, lib):
    assert lib.svo_mutant_id() == 0
    pin(lib)
