"""The CPU oracle against its pins (values printed on the pages, closed forms,
invariants, brute force, an independent library routine)."""
import pytest

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin):
    pin()
