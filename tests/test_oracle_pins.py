"""The oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

import pins


@pytest.mark.parametrize("check", pins.ORACLE_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(orc, check):
    check(orc)


@pytest.mark.parametrize("check", pins.GOLDEN_CHECKS, ids=lambda c: c.__name__)
def test_page_example(orc, golden, check):
    check(orc, golden)


def test_waste_and_sizes(golden):
    pins.check_waste_and_sizes(golden)
