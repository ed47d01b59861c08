"""The oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

import oracle_pin_checks as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(orc, check):
    check(orc)
