"""The CPU oracle against its pins (no GPU needed)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_fixture_matches_printed_rule():
    # the fixture restates "row b scales rows 32*b up to 32*b+32"
    for K, k, b in oracle_pins.read_scale_row_fixture():
        assert 0 <= k < K
        assert 32 * b <= k < 32 * b + 32
