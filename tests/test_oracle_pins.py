"""The CPU oracle against the pages' printed values, closed forms, library
routines and brute force (see tests/oracle_pins.py for each pin's source)."""
import pytest

from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()
