"""Planted mistakes in the oracle must each be caught by at least one pin.

Each mutant is the oracle compiled with one deliberate error (a dropped term, a
wrong sign or index, a transposed operand, an off-by-one mask); see ORACLE_MUTANT
in oracle/oracle.c. This shows the pins are strong enough to trust the oracle.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = {
    1: "softmax Jacobian Delta term dropped",
    2: "interleaved instead of contiguous GQA head groups",
    3: "sliding window one key too wide",
    4: "scale dropped from dK",
    5: "max dropped from LSE",
    6: "ds used in place of p for dV",
    7: "causal diagonal excluded",
    8: "V used in place of K for dQ",
    9: "merge weights with the sign of the exponent flipped",
    10: "merge without the largest lse factored out",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m].replace(" ", "_"))
def test_mutant_is_caught(tmp_path, mutant):
    path = oracle.build(mutant=mutant, out=os.path.join(str(tmp_path), f"liboracle_m{mutant}.so"))
    orc = oracle.Oracle(path)
    assert orc.mutant == mutant
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError) as e:
            caught.append((pin.__name__, str(e)[:80]))
    assert caught, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"
