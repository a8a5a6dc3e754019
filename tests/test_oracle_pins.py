"""The oracle against its pins (closed forms, hand-worked fixtures, library
routines, brute force, Monte-Carlo).  CPU only."""
import pytest

from oracle import pariskv as o
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(o)
