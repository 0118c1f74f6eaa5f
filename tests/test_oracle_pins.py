"""The CPU oracle against the pages' printed values, closed forms and exact
computations (see ``oracle_pins.py`` for what each pin checks)."""
import pytest

from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, oracle, tmp_path):
    pin(oracle, tmp_path)
