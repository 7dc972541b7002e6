"""The oracle against its pins (CPU only)."""
import pytest

from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS,
                         ids=[p.__name__ for p in oracle_pins.ALL_PINS])
def test_pin(pin):
    pin()
