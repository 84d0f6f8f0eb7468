"""Helpers shared by the GPU parity tests (test code only)."""

from __future__ import annotations

import numpy as np

# Tolerances for bf16 inputs with fp32 accumulation against the fp64 oracle.
O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bfloat16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def o_tolerance(o_ref: np.ndarray) -> np.ndarray:
    """Per-element bound on |O_gpu - O_ref|: 1e-2, or one bf16 ulp of the exact
    value where that ulp is larger (|O| >= 2): a bf16 output cannot be closer to
    the exact value than faithful rounding."""
    return np.maximum(O_MAX_ABS, bf16_ulp(o_ref))


def to_device(bits: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def from_device(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """The exact values as the bf16 output format stores them (RNE)."""
    from fa_inputs import bf16_bits_to_float32, round_to_bf16_bits
    return bf16_bits_to_float32(round_to_bf16_bits(x)).astype(np.float64)


def check_parity(o_gpu, lse_gpu, o_ref, lse_ref, label=""):
    """Assert the tolerances; return (max|dO|, mean|dO| vs bf16(O_ref), max|dLSE|).

    * every element: |O_gpu - O_ref| <= max(1e-2, bf16 ulp of O_ref);
    * mean over elements: |O_gpu - bf16(O_ref)| <= 1e-3 -- the mean error of
      the computation, measured against the exact result in the output's own
      format (rounding the exact O to bf16 alone costs up to ~8.5e-4 in mean
      when |O| ~ 1, which would otherwise eat the whole budget);
    * LSE (fp32 output): |LSE_gpu - LSE_ref| <= 1e-3 everywhere.
    """
    err = np.abs(o_gpu - o_ref)
    assert np.isfinite(o_gpu).all() and np.isfinite(lse_gpu).all(), f"{label}: non-finite output"
    bad = err > o_tolerance(o_ref)
    assert not bad.any(), (f"{label}: {int(bad.sum())} O elements beyond tolerance; "
                           f"max err {err.max():.3e}")
    mean_err = float(np.abs(o_gpu - round_bf16(o_ref)).mean())
    assert mean_err <= O_MEAN_ABS, (f"{label}: mean |O - bf16(O_ref)| {mean_err:.3e} "
                                    f"(vs unrounded {err.mean():.3e})")
    el = np.abs(lse_gpu - lse_ref).max()
    assert el <= LSE_MAX_ABS, f"{label}: max |dLSE| {el:.3e}"
    return float(err.max()), mean_err, float(el)
