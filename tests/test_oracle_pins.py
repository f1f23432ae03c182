"""The CPU oracle against brute force, closed forms, invariants and a library
BLAS (no GPU).  The checks themselves live in oracle_pins.py."""
import pytest

import oracle
from tests import oracle_pins as pins


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(o, check):
    check(o)
