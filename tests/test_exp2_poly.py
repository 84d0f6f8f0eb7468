"""The FMA-pipe exp2 of the backward kernel, checked on the CPU.

The kernel's coefficients must be the ones exp2_poly_fit.py derives (Remez,
relative error), and the kernel's steps -- clamp, round to the nearest
integer with the 1.5*2^23 addend, cubic in fused multiply-adds, exponent add
on the bit pattern -- emulated here in fp32 must stay within the stated
relative error bound of exp2 on the whole range the kernel feeds it.
"""

from __future__ import annotations

import os
import re

import numpy as np

from exact_tiled_attention_09_gb300 import exp2_poly_fit

KERNEL = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "exact_tiled_attention_09_gb300", "csrc", "fa_bwd_kernel.cuh")


def _kernel_coefficients():
    text = open(KERNEL).read()
    return [float(np.float32(float(re.search(rf"EXP2_C{i} = ([0-9.eE+-]+)f;", text).group(1))))
            for i in range(4)]


def _fma32(a, b, c):
    # a*b is exact in float64 for float32 inputs; one rounding to float32
    return (a.astype(np.float64) * b + c).astype(np.float32)


def emulate(x):
    x = np.maximum(np.asarray(x, np.float32), np.float32(-126.0))
    t = (x + np.float32(12582912.0)).astype(np.float32)
    n = (t - np.float32(12582912.0)).astype(np.float32)
    f = _fma32(n, np.float32(-1.0), x)
    c0, c1, c2, c3 = (np.float32(c) for c in _kernel_coefficients())
    q = _fma32(f, c3, c2)
    q = _fma32(q, f, c1)
    q = _fma32(q, f, c0)
    bits = (q.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << 23))
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def test_kernel_coefficients_match_the_fit():
    assert _kernel_coefficients() == exp2_poly_fit.fp32_coefficients()


def test_relative_error_bound_over_the_normal_range():
    x = np.concatenate([np.linspace(-125.9, 0.5, 400001, dtype=np.float32),
                        np.float32(-np.arange(0, 126, 0.5))])
    y = emulate(x).astype(np.float64)
    rel = np.abs(y / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() <= 8e-5, rel.max()
    assert exp2_poly_fit.max_relative_error(_kernel_coefficients()) <= 8e-5


def test_underflow_and_minus_infinity_stay_tiny_and_positive():
    y = emulate(np.array([-np.inf, -1e30, -200.0, -126.6, -126.0], np.float32))
    assert np.all(np.isfinite(y)) and np.all(y >= 0) and np.all(y < 2.0 ** -125)
