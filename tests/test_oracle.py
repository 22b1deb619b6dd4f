"""The fp64 oracle against its pins (CPU only)."""
import pytest

import oracle
from tests import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.oracle)


def test_golden_table_matches_mpmath():
    """The stored table itself, re-derived at high precision where mpmath exists."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 30
    for x, Phi, sig in pins.load_activation_table():
        assert abs(float(mp.ncdf(x)) - Phi) < 1e-16
        assert abs(float(1 / (1 + mp.exp(-x))) - sig) < 1e-16
