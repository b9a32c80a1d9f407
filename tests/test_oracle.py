"""The fp64 oracle against its pins (values the pages print, closed forms, invariants,
library special cases and brute force). CPU only."""
import pytest

import oracle
from tests import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_rejects_empty_and_bad_arguments(orc):
    import numpy as np

    with pytest.raises(RuntimeError):
        orc.online_state(np.zeros(2), np.zeros((3, 2)), np.zeros((3, 2)), 0, 3, 1.0, block=0)
    with pytest.raises(RuntimeError):
        orc.attention_online(np.zeros((1, 2)), np.zeros((3, 2)), np.zeros((3, 2)), 1.0, block=0)
