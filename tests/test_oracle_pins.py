"""The fp64 oracle checked against what the pages and the mathematics fix
(CPU only).  See tests/oracle_pins.py for what each pin asserts and why."""
import json
import math
import os

import pytest

import oracle
from tests import oracle_pins

ORC = oracle._get()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(ORC)


def test_threads_do_not_change_results():
    """Splitting rows over threads must not change a single bit."""
    import numpy as np
    r = np.random.default_rng(3)
    q, k, v = (r.standard_normal((2, 3, 70, 16)) for _ in range(3))
    for causal in (False, True):
        o1, l1 = ORC.attention(q, k, v, 0.25, causal, nthreads=1)
        o4, l4 = ORC.attention(q, k, v, 0.25, causal, nthreads=4)
        assert np.array_equal(o1, o4) and np.array_equal(l1, l4)


def test_bad_arguments_rejected():
    import numpy as np
    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(ValueError):
        ORC.attention(q, q, np.zeros((1, 1, 5, 2)), 1.0)
    with pytest.raises(RuntimeError):
        ORC.attention_rows(q, q, q, 1.0, False, [0], [4])   # row out of range
    with pytest.raises(RuntimeError):
        ORC.probabilities(q, q, 1.0, False, bh=1)            # head out of range


def test_empty_sequence():
    import numpy as np
    q = np.zeros((1, 2, 0, 8))
    o, lse = ORC.attention(q, q, q, 1.0, True)
    assert o.shape == (1, 2, 0, 8) and lse.shape == (1, 2, 0)
