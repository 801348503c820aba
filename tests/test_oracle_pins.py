"""The committed fp64 oracle passes every pin (hand-worked examples, closed
forms, library routines, pure-Python brute force)."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.default())


def test_bad_arguments_rejected():
    import numpy as np
    W = np.zeros((100, 4), dtype=np.float16)
    with pytest.raises(ValueError):
        oracle.quantize_pack(W, group=128)        # K % group != 0
    with pytest.raises(ValueError):
        oracle.quantize_pack(np.zeros((12, 4), dtype=np.float16), group=12)  # group % 8
