"""The oracle against what the pages and mathematics fix (CPU only)."""
import pytest

import oracle_pins
from oracle.oracle import default


@pytest.fixture(scope="module")
def orc():
    return default()


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_bf16_widening_is_exact(orc):
    # 0x3F80 = 1.0, 0xC000 = -2.0, 0x3E20 = 0.15625, 0x7F7F = largest finite bf16
    assert orc.bf16_value(0x3F80) == 1.0
    assert orc.bf16_value(0xC000) == -2.0
    assert orc.bf16_value(0x3E20) == 0.15625
    assert orc.bf16_value(0x7F7F) == float.fromhex("0x1.fep127")
