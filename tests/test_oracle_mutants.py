"""Each deliberate mistake planted in the oracle (compile-time variants, CPU only) must
fail at least one pin: the pins are strong enough to catch a dropped term, a wrong index,
a wrong sign or scale."""

import pytest

import oracle
import pins


@pytest.mark.parametrize("mutant", sorted(oracle.MUTANTS), ids=lambda m: oracle.MUTANTS[m])
def test_pins_catch_planted_mistake(mutant):
    orc = oracle.load(mutant)
    assert orc.lib.oracle_mutant_id() == mutant
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            check(orc)
        except (AssertionError, ValueError):
            caught.append(check.__name__)
    assert caught, f"no pin catches mutant {mutant}: {oracle.MUTANTS[mutant]}"
