"""The oracle against its pins (hand-worked fixtures, library routines,
closed forms, invariants).  CPU only."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=[c.__name__ for c in P.ALL_CHECKS])
def test_pin(orc, check):
    check(orc)
