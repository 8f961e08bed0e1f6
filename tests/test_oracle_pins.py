"""The oracle against its pins: a library routine, closed forms, invariants, fixtures."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_oracle_is_not_a_mutant(orc):
    assert orc.mutant == 0
