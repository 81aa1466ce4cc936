"""The CPU oracle against its pins (no GPU needed)."""
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def O():
    return oracle.default()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(O, pin):
    if pin in (pins.pin_philox_vs_triton, pins.pin_noise_layout):
        pytest.importorskip("triton")
    pin(O)
