"""Coefficients of the polynomial behind the softplus gate of the kernels.

The gate needs softplus(x) = log(1 + e^x) once per channel and token.  The
kernels write it as

    softplus(x) = max(x, 0) + log1p(z),   z = e^{-|x|} in (0, 1],

an identity for every real x, and evaluate log1p(z) = z * P(z), where P is a
degree-9 polynomial fitted to log1p(z) / z (which is 1 at z = 0 and ln 2 at
z = 1) by least squares on 4000 Chebyshev nodes of [0, 1], in double
precision, then rounded to fp32.  The nearest singularity of log1p(z) / z is
at z = -1, so the fit converges geometrically; at degree 9 the fp32
evaluation (Horner with fused multiply-adds, then the product with z) is
within 2 units in the last place of log1p(z) on all of [0, 1], which
``tests/test_softplus_poly.py`` checks against double-precision log1p.

Run as a script to print the C++ initialiser that ``kda_device.cuh`` holds.
"""

from __future__ import annotations

import numpy as np

DEGREE = 9
NODES = 4000


def coefficients() -> np.ndarray:
    """fp32 coefficients c[0..DEGREE] of P(z) = sum c[i] z^i."""
    k = np.arange(NODES)
    z = 0.5 - 0.5 * np.cos((2 * k + 1) * np.pi / (2 * NODES))
    f = np.log1p(z) / z
    vander = np.vander(z, DEGREE + 1, increasing=True)
    c, *_ = np.linalg.lstsq(vander, f, rcond=None)
    return c.astype(np.float32)


def _hex(c: np.float32) -> str:
    mant, exp = float(c).hex().split("p")
    mant = mant.rstrip("0").rstrip(".")
    return f"{mant}p{exp}f"


def c_initialiser() -> str:
    return ", ".join(_hex(c) for c in coefficients())


if __name__ == "__main__":
    print(c_initialiser())
