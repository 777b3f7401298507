"""The oracle against its pins (CPU only)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(oracle_lib, pin):
    pin(oracle_lib)


def test_oracle_rejects_bad_shapes(oracle_lib):
    import numpy as np
    with pytest.raises(ValueError):
        oracle_lib.trimul(np.zeros(3 * 10 * 1, np.uint16), 1, 1, 10, 3)  # C % NH != 0
    with pytest.raises(ValueError):
        oracle_lib.trimul_rows(np.zeros(3 * 8, np.uint16), 1, 1, 8, 1, np.array([[0, 0, 1]]))


def test_oracle_threads(oracle_lib):
    assert oracle_lib.num_threads() >= 1
