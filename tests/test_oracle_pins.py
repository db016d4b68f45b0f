"""The CPU oracle against facts other than itself (no GPU needed)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin, oracle_handle):
    if pin.__name__ == "pin_symbolic_small_T":
        pytest.importorskip("sympy")
    pin(oracle_handle)
