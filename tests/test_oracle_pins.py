"""The CPU oracle against facts that do not come from itself (CPU only)."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


@pytest.mark.parametrize("name", sorted(oracle_pins.ALL_CHECKS))
def test_pin(o, name):
    oracle_pins.ALL_CHECKS[name](o)
