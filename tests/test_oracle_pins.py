"""The oracle against what the pages and mathematics fix (CPU only)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_relu_gradients_finite_difference(orc):
    import oracle
    oracle_pins.pin_gradients_finite_difference(orc, act=oracle.ACT_RELU)


def test_oracle_threads(orc):
    assert orc.num_threads() >= 1
