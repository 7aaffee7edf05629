"""The fp64 oracle against closed forms, group laws, independent formulations,
library routines and brute force (see tests/oracle_pins.py for what each pins)."""
import pytest

import oracle as O
from tests import oracle_pins as P


@pytest.fixture(scope="module")
def orc():
    return O.default()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)
