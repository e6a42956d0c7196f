"""The CPU oracle against what the pages and the mathematics fix (CPU only).

The checks live in tests/oracle_pins.py so the same pins can be run against
deliberately broken oracle builds (test_oracle_mutants.py)."""
import pytest

import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_FAST, ids=lambda f: f.__name__)
def test_pin(check, oracle_lib):
    check(oracle_lib)


@pytest.mark.parametrize("check", pins.ALL_MC, ids=lambda f: f.__name__)
def test_monte_carlo(check, oracle_lib):
    check(oracle_lib)
