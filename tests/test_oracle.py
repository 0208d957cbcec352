"""The fp64 oracle against its pins (no GPU)."""
import pytest

import oracle_pins
from oracle import ra_oracle


@pytest.fixture(scope="module")
def O():
    return ra_oracle.get()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(O, pin):
    pin(O)


def test_rejects_bad_arguments(O):
    import numpy as np
    q = np.zeros((1, 6, 2))
    with pytest.raises(ValueError):
        O.ring(q, q, q, P=4)  # 4 does not divide 6
    with pytest.raises(ValueError):
        O.ring(q, q, q, P=2, t0=1, t1=3)
