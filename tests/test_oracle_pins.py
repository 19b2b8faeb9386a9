"""The CPU oracle against what the pages and mathematics fix (no GPU)."""
import pytest

from oracle import moe_oracle
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(moe_oracle)
