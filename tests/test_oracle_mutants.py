"""Mutation test of the oracle's pins: each planted mistake (compiled into the
oracle with LT_ORACLE_MUTANT=k, on the CPU) must fail at least one pin."""

import pytest

import oracle
import pins

MUTANTS = {
    1: "eps added outside the square root",
    2: "sum of squares used instead of the mean",
    3: "W read transposed",
    4: "first shared partial dropped",
    5: "routed partials read with the wrong layout",
    6: "norm weight dropped",
    7: "shared partials read with the wrong layout",
    8: "W row taken relative to the column range",
    9: "squares of partials summed instead of the square of the sum",
    10: "no-norm branch still normalizes",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda k: f"m{k}")
def test_pins_catch_planted_mistake(tmp_path, mutant):
    so = oracle.build(tmp_path / f"liblt_oracle_m{mutant}.so", mutant=mutant)
    lib = oracle.load(so)
    assert lib.lt_oracle_mutant_id() == mutant
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {mutant}: {MUTANTS[mutant]}"
