"""The CPU oracle against facts the pages and the mathematics fix (no GPU)."""
import pytest

import oracle
from tests import oracle_pin_checks as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle.default())
