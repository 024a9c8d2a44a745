"""The oracle against facts other than its own formula (no GPU needed)."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin_holds(pin):
    assert pin(oracle.lib()) == []
