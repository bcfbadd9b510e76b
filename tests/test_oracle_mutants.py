"""Each planted mistake in the oracle (a dropped term, a wrong index, a wrong
grouping, a missing scale, the wrong log base ...) must fail at least one
pin: evidence that the pins pin the oracle, not just run it."""

import pytest

import oracle
import pins


@pytest.mark.parametrize("mutant", sorted(oracle.MUTANTS), ids=lambda m: oracle.MUTANTS[m])
def test_mutant_is_caught(mutant):
    orc = oracle.Oracle(mutant)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {mutant}: {oracle.MUTANTS[mutant]}"
