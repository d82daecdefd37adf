"""Planted mistakes in the oracle must each fail at least one pin.

Each mutant is the oracle compiled with -DGDN_ORACLE_MUTANT=k, which swaps
one line for a plausible mistake: reversed conv taps (1), history order
flipped (2), decay dropped (3), sign of the delta flipped (4), state read
transposed (5), grouped heads mapped h mod H_k (6), output read before the
rank-one update (7), k not normalised (8), dt_bias dropped (9), commit path
applied leaf first (10), commit window from the parent (11), b and a swapped
(12), SiLU dropped (13), q not normalised (14).  CPU only.
"""
import pytest

import oracle as O
import oracle_pins as P

MUTANTS = list(range(1, 15))


@pytest.mark.parametrize("mutant", MUTANTS)
def test_mutant_is_caught(mutant):
    orc = O.Oracle(mutant=mutant)
    caught = []
    for check in P.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            caught.append(check.__name__)
    assert caught, f"mutant {mutant} passed every pin"
