"""The kernels' softplus (CPU): the polynomial in the device header matches its
generator, and its fp32 evaluation is within 2 ulp of log1p on [0, 1] and of
the double-precision softplus over the gate's input range.

The device code evaluates log1p(z) = z * P(z) by Horner's rule with fused
multiply-adds; here each fp32 fused multiply-add is emulated in double
precision (the product of two fp32 numbers is exact in double), which can
differ from a true fused multiply-add by one rounding in rare cases; the
2-ulp bound leaves room for that."""

import os
import re
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "linear_attention_speculative_kda_gb300", "csrc")
sys.path.insert(0, CSRC)

import softplus_poly  # noqa: E402


def header_coefficients() -> np.ndarray:
    text = open(os.path.join(CSRC, "kda_device.cuh")).read()
    body = re.search(r"float softplus\(float x\) \{.*?constexpr float c\[10\] = \{(.*?)\};",
                     text, re.S).group(1)
    vals = [float.fromhex(t.strip().rstrip("f")) for t in body.split(",")]
    return np.array(vals, dtype=np.float32)


def fma32(a, b, c):
    return (np.asarray(a, np.float64) * np.asarray(b, np.float64)
            + np.asarray(c, np.float64)).astype(np.float32)


def log1p32(z, c):
    z = np.asarray(z, np.float32)
    r = np.full(z.shape, c[-1], np.float32)
    for ci in c[-2::-1]:
        r = fma32(r, z, ci)
    return (z.astype(np.float64) * r.astype(np.float64)).astype(np.float32)


def softplus32(x, c):
    """The device formula with an exactly rounded z = e^{-|x|}."""
    x = np.asarray(x, np.float32)
    z = np.exp(-np.abs(x.astype(np.float64))).astype(np.float32)
    l = log1p32(z, c)
    sp = np.where(x > 0, (x.astype(np.float64) + l.astype(np.float64)).astype(np.float32), l)
    return np.where(x > 20, x, sp)


def ulps(got, want):
    want32 = np.abs(want).astype(np.float32)
    return np.abs(got.astype(np.float64) - want) / np.spacing(want32).astype(np.float64)


def test_header_matches_generator():
    hdr = header_coefficients()
    gen = softplus_poly.coefficients()
    assert hdr.shape == gen.shape == (softplus_poly.DEGREE + 1,)
    # equal, or one fp32 step apart if the host's LAPACK rounds differently
    steps = np.abs(hdr.view(np.int32).astype(np.int64) - gen.view(np.int32).astype(np.int64))
    assert steps.max() <= 1


def test_log1p_within_two_ulp():
    c = header_coefficients()
    z = np.concatenate([np.linspace(0, 1, 400001, dtype=np.float32),
                        np.float32(2.0) ** -np.arange(1, 120, dtype=np.float32)])
    z = z[z > 0]
    got = log1p32(z, c)
    want = np.log1p(z.astype(np.float64))
    assert ulps(got, want).max() <= 2.0
    assert log1p32(np.float32(1.0), c) == np.float32(np.log(2.0))  # P(1) = ln 2
    assert log1p32(np.float32(0.0), c) == 0.0


def test_softplus_over_gate_range():
    c = header_coefficients()
    x = np.linspace(-30, 30, 600001, dtype=np.float32)
    got = softplus32(x, c)
    x64 = x.astype(np.float64)
    want = np.where(x64 > 20, x64, np.log1p(np.exp(x64)))
    assert ulps(got, want).max() <= 2.0
    # the identity's two branches meet without a step at x = 0
    assert softplus32(np.float32(0.0), c) == np.float32(np.log(2.0))
