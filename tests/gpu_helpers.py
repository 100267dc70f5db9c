"""Shared helpers for the GPU parity tests."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances: max-abs error on the 16-bit output O and on the fp32 LSE
# (fp32 accumulation inside the kernels; P is rounded to 16 bits before P V).
O_TOL = 2e-2
LSE_TOL = 1e-3


def dev(*ts):
    return [t.cuda().contiguous() for t in ts]


def max_abs_err(actual, expected):
    a = actual.detach().to("cpu", torch.float64).numpy() if hasattr(actual, "detach") else np.asarray(actual)
    e = expected.detach().to("cpu", torch.float64).numpy() if hasattr(expected, "detach") else np.asarray(expected)
    assert a.shape == e.shape, (a.shape, e.shape)
    if a.size == 0:
        return 0.0, None
    same = a == e  # includes equal infinities (e.g. LSE = -inf of an empty sequence)
    bad = ~same & ~(np.isfinite(a) & np.isfinite(e))
    if np.any(bad):
        return float("inf"), tuple(int(x) for x in np.argwhere(bad)[0])
    with np.errstate(invalid="ignore"):
        d = np.where(same, 0.0, np.abs(a - e))
    idx = np.unravel_index(int(np.argmax(d)), d.shape)
    return float(d[idx]), tuple(int(x) for x in idx)


def assert_close(actual, expected, tol, what=""):
    err, where = max_abs_err(actual, expected)
    assert err <= tol, f"{what}: max abs err {err:.3e} at {where} > {tol:.1e}"
    return err
