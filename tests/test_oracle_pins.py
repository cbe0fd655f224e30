"""The CPU oracle against what the pages and mathematics fix (no GPU needed)."""
import pytest

import os, sys
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import oracle_pins as pins  # noqa: E402


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check()
