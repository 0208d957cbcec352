"""Each planted mistake in the oracle must fail at least one pin (no GPU).

The mistakes are compiled into separate copies of the oracle via the
``ORA_MUTANT`` switch: o not rescaled (1), l not rescaled (2), per-block
normalise-then-average (3), 1/d instead of 1/sqrt(d) (4), sign flip in the
exponent (5), K used in place of V (6), a strict causal mask that hides the
query's own key (7), the backward's row term D dropped from dS (8).
"""
import numpy as np
import pytest

import oracle_pins
from oracle import ra_oracle

MUTANTS = [1, 2, 3, 4, 5, 6, 7, 8]


@pytest.mark.parametrize("mutant", MUTANTS)
def test_mutant_is_caught(mutant, tmp_path_factory):
    out = tmp_path_factory.mktemp(f"m{mutant}")
    O = ra_oracle.Oracle(mutant=mutant, outdir=out)
    assert O.mutant == mutant
    caught = []
    with np.errstate(all="ignore"):
        for pin in oracle_pins.ALL_PINS:
            try:
                pin(O)
            except (AssertionError, ValueError, FloatingPointError):
                caught.append(pin.__name__)
    assert caught, f"mutant {mutant} passed every pin"
