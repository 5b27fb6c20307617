"""The CPU oracle against facts fixed by the pages and by the mathematics
(see oracle_pins.py for the list and citations). CPU only."""
import pytest

import oracle as O
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(O.default())
