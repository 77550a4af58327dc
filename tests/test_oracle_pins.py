"""The oracle against facts that do not come from it (see tests/pins.py)."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(oracle, pin):
    pin(oracle)


def test_oracle_rejects_bad_arguments(oracle):
    import numpy as np
    with pytest.raises(ValueError):
        oracle.topk(np.zeros((2, 3), np.float32), 4)       # K > cols
    with pytest.raises(ValueError):
        oracle.topk(np.zeros((2, 3), np.float32), 0)
    with pytest.raises(ValueError):
        oracle.preprocess(np.zeros((1, 4, 6), np.uint8), 2, 4, 0, 3)
    with pytest.raises(ValueError):
        oracle.inner_box(0, 1, 1, 1, True)
