"""Planted mistakes: build the oracle with one deliberate error at a time
(CPU only) and check that at least one pin of test_oracle.py fails on it."""
import pytest

import oracle
from test_oracle import ALL_PINS

MUTANTS = {
    1: "B nibble order swapped",
    2: "32-element scale blocks",
    3: "last k term dropped",
    4: "E4M3 bias 8",
    5: "rounding through fp32",
    6: "E2M1 subnormal read as 1.0",
    7: "E2M1 sign from the wrong bit",
    8: "scale atoms ordered row-block fastest",
    9: "fp16 ties away from zero",
    10: "every sum declared exact",
    11: "exactness bound one bit past fp64",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m])
def test_some_pin_catches_mutant(mutant):
    o = oracle.Oracle(oracle.build(mutant=mutant))
    assert o.lib.oracle_mutant_id() == mutant
    caught = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches planted mistake {mutant}: {MUTANTS[mutant]}"
