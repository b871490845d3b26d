"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

from oracle import lg_oracle
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(lg_oracle)
