"""The fp64 oracle against library routines, closed forms and invariants.

CPU only.  A second test builds the oracle with each planted mistake
(ORACLE_MUTANT=n) and checks that at least one pin fails for every one of
them, so the pins are known to bite.
"""
import os
import tempfile

import pytest

from oracle import oracle as O
from tests.oracle_pins import PINS

N_MUTANTS = 16


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(O.load())


def test_every_planted_mistake_is_caught():
    caught = {}
    with tempfile.TemporaryDirectory() as tmp:
        for n in range(1, N_MUTANTS + 1):
            path = os.path.join(tmp, f"liboracle_m{n}.so")
            O.build(path, mutant=n, force=True)
            lib = O.load(path)
            failing = []
            for pin in PINS:
                try:
                    pin(lib)
                except (AssertionError, ValueError) as e:  # noqa: PERF203
                    failing.append(pin.__name__)
            caught[n] = failing
    missed = [n for n, f in caught.items() if not f]
    assert not missed, f"planted mistakes not caught by any pin: {missed}; caught: {caught}"
