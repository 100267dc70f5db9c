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


# Gradient tolerance of the backward tests: the kernel rounds P and dS to 16
# bits before their products and accumulates in fp32, so an element of dQ, dK
# or dV carries a relative error of a few 2^-9 of the magnitudes that meet in
# its sum.
GRAD_TOL = 2e-2
FRO_TOL = 1e-2


def assert_grad_close(got, ref, what):
    """max |g - ref| <= 2e-2 max(1, max |ref|) and ||g - ref|| <= 1e-2
    max(||ref||, sqrt(n)) (the Frobenius floor is an O(1) scale per element:
    an exactly zero reference only meets rounding noise)."""
    g = got.double().numpy() if hasattr(got, "numpy") else np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = float(np.max(np.abs(g - r))) if g.size else 0.0
    bound = GRAD_TOL * max(1.0, float(np.max(np.abs(r))) if r.size else 0.0)
    fro = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), np.sqrt(max(r.size, 1))))
    assert err <= bound and fro <= FRO_TOL, f"{what}: max err {err:.3e} (bound {bound:.3e}), rel fro {fro:.3e}"
