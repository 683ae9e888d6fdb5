"""The float64 oracle against what the pages and mathematics fix (CPU only)."""
import pytest

import oracle
from tests import _pins


@pytest.mark.parametrize("pin", _pins.PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle)


def test_thread_count_does_not_change_result():
    import numpy as np
    rng = np.random.default_rng(0)
    T, H, dk, dv = 17, 5, 4, 3
    q, k, v, g, b = _pins._rand_problem(rng, T, H, dk, dv)
    cu = np.array([0, 7, 7, 17])
    S0 = rng.standard_normal((3, H, dk, dv))
    o1, S1 = oracle.prefill(q, k, v, g, b, S0=S0, cu_seqlens=cu, nthreads=1)
    o4, S4 = oracle.prefill(q, k, v, g, b, S0=S0, cu_seqlens=cu, nthreads=4)
    np.testing.assert_array_equal(o1, o4)
    np.testing.assert_array_equal(S1, S4)


def test_rejects_bad_cu_seqlens():
    import numpy as np
    x = np.zeros((4, 1, 2))
    with pytest.raises(ValueError):
        oracle.prefill(x, x, x, x, np.zeros((4, 1)), cu_seqlens=[0, 3, 2, 4])
    with pytest.raises(ValueError):
        oracle.prefill(x, x, x, x, np.zeros((4, 1)), cu_seqlens=[0, 3])
