"""Each planted mistake in the oracle (built with -DORACLE_MUTANT=n) must fail a pin."""
import pytest

import oracle
from tests import oracle_pins


@pytest.mark.parametrize("mutant", range(1, oracle.N_MUTANTS + 1))
def test_mutant_is_caught(mutant):
    orc = oracle.Oracle(mutant)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} passed every pin"
