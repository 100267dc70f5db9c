"""The fp64 oracle against its pins (library routines, closed forms, invariants)."""
import numpy as np
import pytest
import torch

import oracle
from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(oracle.get())


def test_widening_is_exact():
    """The oracle receives exactly the 16-bit values the kernels see."""
    for dt in (torch.float16, torch.bfloat16):
        x = torch.randn(1000, generator=torch.Generator().manual_seed(3)).to(dt)
        w = oracle._f64(x)
        assert w.dtype == np.float64
        assert np.array_equal(w, x.to(torch.float32).numpy().astype(np.float64))


def test_bad_arguments_raise():
    q = torch.zeros(1, 4, 8, dtype=torch.float64)
    with pytest.raises(ValueError):
        oracle.attention(q, torch.zeros(1, 4, 9, dtype=torch.float64), torch.zeros(1, 4, 9, dtype=torch.float64),
                         False, 1.0)
    with pytest.raises(ValueError):
        oracle.attention(q, q, q, False, 1.0, rows=[4])  # row out of range
    with pytest.raises(ValueError):  # every partition empty cannot be merged
        oracle.splitkv_merge(np.zeros((1, 2, 8)), np.full((1, 2), -np.inf), np.zeros((1, 2)))


def test_threads_do_not_change_results():
    g = torch.Generator().manual_seed(9)
    q, k, v = (torch.randn(6, 33, 16, generator=g, dtype=torch.float64) for _ in range(3))
    a = oracle.attention(q, k, v, True, 0.3, nthreads=1)
    b = oracle.attention(q, k, v, True, 0.3, nthreads=4)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
