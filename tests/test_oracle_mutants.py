"""Each planted mistake in the oracle (dropped term, wrong index, lost
initial value, wrong sign, off-by-one, transposed operand, single-precision
bias sum) must be caught by at least one pin. The mistakes live in builds of
the oracle compiled with ORACLE_MUTANT set; the real build never sets it."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("mutant", oracle.MUTANTS)
def test_mutant_is_caught(mutant):
    orc = oracle.Oracle(f"mutant{mutant}")
    assert orc._lib.oracle_mutant() == mutant
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} passed every pin"
