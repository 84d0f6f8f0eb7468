"""The oracle pins must reject plausible mistakes.

Each mutant is a deliberately broken copy of the oracle's definition (in
matrix form, CPU only).  The test runs the same pin checks used on the real
oracle and asserts that at least one of them fails for the mutant, while
all of them pass for the unmodified definition.
"""

from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
from fa_inputs import bf16_bits_to_float32, make_custom
from tests.test_oracle_pins import _brute


def _definition(q, k, v, scale, causal, mutation=None):
    L = q.shape[0]
    s = scale * (q @ k.T)
    if mutation == "transposed_scores":
        s = scale * (k @ q.T)
    if mutation == "dropped_scale":
        s = q @ k.T
    allowed = np.tril(np.ones((L, L), dtype=bool)) if causal else np.ones((L, L), bool)
    if mutation == "causal_off_by_one" and causal:
        allowed = np.tril(np.ones((L, L), dtype=bool), -1)
        allowed[0, 0] = True
    s = np.where(allowed, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m) if mutation != "sign_flip" else np.where(allowed, np.exp(m - s), 0.0)
    z = e.sum(axis=1, keepdims=True)
    p = e / z
    if mutation == "unnormalised":
        p = e
    o = p @ v
    if mutation == "probs_transposed":
        o = p.T @ v
    lse = (m + np.log(z))[:, 0]
    if mutation == "lse_without_max":
        lse = np.log(z)[:, 0]
    return o, lse


def _pins_pass(fn) -> bool:
    """The pin checks of test_oracle_pins, applied to a candidate oracle."""
    f = lambda b: bf16_bits_to_float32(b).astype(np.float64)[0, 0]
    for causal in (False, True):
        for L in (5, 9):
            qb, kb, vb = make_custom(1, 1, L, 4, 300 + L, 2.0, 2.0, 1.0)
            q, k, v = f(qb), f(kb), f(vb)
            o, lse = fn(q, k, v, 0.6, causal)
            o_b, lse_b = _brute(q, k, v, 0.6, causal)
            if np.abs(o - o_b).max() > 1e-13 or np.abs(lse - lse_b).max() > 1e-13:
                return False
        # closed form: scale 0 gives the mean of the allowed rows and ln(count)
        o, lse = fn(q, k, v, 0.0, causal)
        for i in range(q.shape[0]):
            n = i + 1 if causal else q.shape[0]
            if np.abs(o[i] - v[:n].mean(axis=0)).max() > 1e-14 or abs(lse[i] - math.log(n)) > 1e-14:
                return False
    return True


def test_unmodified_definition_passes_the_pins():
    assert _pins_pass(lambda q, k, v, s, c: _definition(q, k, v, s, c))
    assert _pins_pass(lambda q, k, v, s, c: oracle.attention(q, k, v, s, c))


@pytest.mark.parametrize("mutation", ["transposed_scores", "dropped_scale", "causal_off_by_one",
                                      "sign_flip", "unnormalised", "probs_transposed",
                                      "lse_without_max"])
def test_mutant_is_rejected(mutation):
    assert not _pins_pass(lambda q, k, v, s, c: _definition(q, k, v, s, c, mutation))


# --------------------------------------------------------------------------
# Gradient oracle: each mutant of the backward formulas must fail the pins
# of tests/test_oracle_bwd_pins.py (finite differences and invariants).
# --------------------------------------------------------------------------
def _bwd_definition(q, k, v, dout, scale, causal, mutation=None):
    L = q.shape[-2]
    s = scale * (q @ np.swapaxes(k, -1, -2))
    allowed = np.tril(np.ones((L, L), dtype=bool)) if causal else np.ones((L, L), bool)
    if mutation != "mask_ignored":
        s = np.where(allowed, s, -np.inf)
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    p = e / e.sum(axis=-1, keepdims=True)
    pt = np.swapaxes(p, -1, -2)
    dv = pt @ dout if mutation != "dv_untransposed" else p @ dout
    dp = dout @ np.swapaxes(v, -1, -2)
    rowsum = (dp * p).sum(axis=-1, keepdims=True)
    if mutation == "rowsum_over_keys_axis":
        rowsum = (dp * p).sum(axis=-2, keepdims=True)
    ds = p * (dp - rowsum) if mutation != "dropped_rowsum" else p * dp
    if mutation == "sign_flip":
        ds = p * (rowsum - dp)
    dst = np.swapaxes(ds, -1, -2)
    dq = scale * (ds @ k) if mutation != "dq_transposed" else scale * (dst @ k)
    dk = scale * (dst @ q)
    if mutation == "dk_unscaled":
        dk = dst @ q
    if mutation == "dk_uses_k":
        dk = scale * (dst @ k)
    return dq, dk, dv


def test_unmodified_gradient_definition_passes_the_pins():
    from tests.test_oracle_bwd_pins import pins_pass
    assert pins_pass(lambda *a: _bwd_definition(*a))


@pytest.mark.parametrize("mutation", ["mask_ignored", "dv_untransposed", "rowsum_over_keys_axis",
                                      "dropped_rowsum", "sign_flip", "dq_transposed",
                                      "dk_unscaled", "dk_uses_k"])
def test_gradient_mutant_is_rejected(mutation):
    from tests.test_oracle_bwd_pins import pins_pass
    assert not pins_pass(lambda *a: _bwd_definition(*a, mutation=mutation))
