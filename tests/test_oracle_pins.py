"""The FP64 oracle against closed forms, invariants and brute force (CPU only)."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle.default())


def test_threads_positive():
    assert oracle.threads() >= 1
    assert oracle.threads(3) == 3


def test_bad_arguments_rejected():
    import numpy as np
    with pytest.raises(ValueError):
        oracle.accel(np.zeros((4, 3)), 0.1)
    with pytest.raises(ValueError):
        oracle.accel(np.zeros((4, 4)), 0.1, idx=[4])
    with pytest.raises(ValueError):
        oracle.leapfrog(np.zeros((4, 4)), np.zeros((4, 3)), 0.1, 0.1, -1)
