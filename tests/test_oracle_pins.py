"""The CPU oracle against its pins (closed forms, eq (8) brute force, eq (10)-(12)
composition, special cases, exact invariances).  CPU only."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_rejects_bad_arguments(orc):
    import numpy as np
    import ctypes
    f = np.zeros((1, 1, 4), np.float32)
    A = np.zeros((1, 1), np.float32)
    # size <= 0 is refused with status 1
    rc = orc.lib.ss_oracle_fwd(f.ctypes.data, f.ctypes.data, A.ctypes.data, f.ctypes.data,
                               f.ctypes.data, None, None, None, 1, None,
                               f.ctypes.data, None, 0, 1, 1, 4, 0, 1)
    assert rc == 1
