"""Both CPU oracles -- numpy (cp_oracle.py) and C++ (cp_oracle.cpp through
oracle/cpp.py) -- against the same pins (values printed on the pages, closed
forms, invariants, brute force, an independent library routine)."""
import pytest

import oracle.cp_oracle as numpy_oracle
import oracle.cpp as cpp_oracle
import oracle_pins
from oracle_pins import ALL_PINS

IMPLS = {"numpy": numpy_oracle, "cpp": cpp_oracle}


@pytest.mark.parametrize("impl", sorted(IMPLS))
@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin, impl, monkeypatch):
    monkeypatch.setattr(oracle_pins, "O", IMPLS[impl])
    pin()
