"""Each deliberately broken build of the oracle must fail at least one pin.

The mistakes are planted in the oracle source behind ORACLE_MUTANT (CPU only):
1 window edge off by one, 2 scale dropped, 3 interleaved instead of grouped GQA heads,
4 causal mask dropped, 5 owner map ignored, 6 softmax normaliser over every cached key,
7 query position without the cached prefix, 8 soft-cap applied to the unscaled score,
9 the last of equal maximal logits taken as the greedy index, 10 logit cap without the
division by the cap.
"""
import os

import pytest

import oracle_pins
from oracle.oracle import Oracle, OracleError, build_oracle

MUTANTS = [1, 2, 3, 4, 5, 6, 7, 8, 9, 10]


@pytest.mark.parametrize("mutant", MUTANTS)
def test_mutant_is_caught(tmp_path, mutant):
    path = build_oracle(out=os.path.join(str(tmp_path), f"liboracle_m{mutant}.so"), mutant=mutant)
    orc = Oracle(path)
    assert orc.mutant == mutant
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, OracleError) as e:  # the pin noticed the planted mistake
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} passed every pin"
