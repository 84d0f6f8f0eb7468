"""Helpers shared by the GPU parity tests (test code only)."""

from __future__ import annotations

import math

import numpy as np

# Tolerances for bf16 inputs with fp32 accumulation against the fp64 oracle.
O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3
# Compute allowance of the per-element bound: the error the kernel may make
# before its output is rounded to bf16.  P~ is rounded to bf16 (unit
# roundoff 2^-8) before the P~ V product while the row sum l adds the fp32
# values, so O_ic moves by at most 2^-8 * A_ic with A_ic = sum_j (p_ij / l_i)
# |v_jc| -- attention applied to |V|, which the oracle computes exactly
# (``oracle_forward``).  fp32 accumulation over at most 2^16 keys adds under
# 2^-16 * A_ic.  (A row dominated by one key carries that key's weight
# exactly: the running max makes it exp2(0) = 1.)
O_COMPUTE_ALLOW_REL = 2.0 ** -8 + 2.0 ** -16

# (config, label, max|dO|, mean|dO - bf16(O_ref)|, mean|dO| vs exact, max|dLSE|)
# of every check_parity call that names a configuration, printed as a table
# at the end of the GPU session (tests/conftest.py).
PARITY_LOG: list = []


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bfloat16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def o_tolerance(o_ref: np.ndarray, absv_ref: np.ndarray) -> np.ndarray:
    """Per-element bound on |O_gpu - O_ref|: 1e-2 (the stated tolerance), or,
    where it is larger, the compute allowance a = O_COMPUTE_ALLOW_REL * A
    plus half a bf16 ulp of the value the kernel rounds (|O_ref| + a):
    correct rounding of a result that is itself within a of the exact one."""
    a = O_COMPUTE_ALLOW_REL * np.abs(absv_ref)
    return np.maximum(O_MAX_ABS, 0.5 * bf16_ulp(np.abs(o_ref) + a) + a)


def oracle_forward(q, k, v, scale, causal=False, rows=None):
    """The oracle's (O, LSE) and A = attention applied to |V| (the weighted
    mean of |v| per output element, for the per-element bound)."""
    import oracle
    o, lse = oracle.attention(q, k, v, scale, causal, rows=rows)
    a, _ = oracle.attention(q, k, np.abs(v), scale, causal, rows=rows)
    return o, lse, a


def to_device(bits: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def from_device(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """The exact values as the bf16 output format stores them (RNE)."""
    from fa_inputs import bf16_bits_to_float32, round_to_bf16_bits
    return bf16_bits_to_float32(round_to_bf16_bits(x)).astype(np.float64)


def check_parity(o_gpu, lse_gpu, o_ref, lse_ref, label="", config=None, absv_ref=None):
    """Assert the tolerances; return (max|dO|, mean|dO| vs bf16(O_ref), max|dLSE|).

    * every element: |O_gpu - O_ref| <= o_tolerance(O_ref, A) (``absv_ref``
      = A from ``oracle_forward``; required);
    * mean over elements: |O_gpu - bf16(O_ref)| <= 1e-3 -- the mean error of
      the computation, measured against the exact result in the output's own
      format (rounding the exact O to bf16 alone costs up to ~8.5e-4 in mean
      when |O| ~ 1, which would otherwise eat the whole budget); the mean
      against the unrounded O_ref is logged beside it (``config``);
    * LSE (fp32 output): |LSE_gpu - LSE_ref| <= 1e-3 everywhere.
    """
    assert absv_ref is not None, "check_parity needs A = attention of |V| (oracle_forward)"
    err = np.abs(o_gpu - o_ref)
    assert np.isfinite(o_gpu).all() and np.isfinite(lse_gpu).all(), f"{label}: non-finite output"
    bad = err > o_tolerance(o_ref, np.asarray(absv_ref).reshape(o_ref.shape))
    assert not bad.any(), (f"{label}: {int(bad.sum())} O elements beyond tolerance; "
                           f"max err {err.max():.3e}")
    mean_err = float(np.abs(o_gpu - round_bf16(o_ref)).mean())
    assert mean_err <= O_MEAN_ABS, (f"{label}: mean |O - bf16(O_ref)| {mean_err:.3e} "
                                    f"(vs unrounded {err.mean():.3e})")
    el = float(np.abs(lse_gpu - lse_ref).max())
    assert el <= LSE_MAX_ABS, f"{label}: max |dLSE| {el:.3e}"
    if config is not None:
        PARITY_LOG.append((config, label, float(err.max()), mean_err, float(err.mean()), el))
    return float(err.max()), mean_err, el


# Gradients (backward pass).  Per head and per gradient tensor G, against the
# exact fp64 gradient:
#   max |G - G_ref|      <= GRAD_MAX_REL * max |G_ref| + GRAD_ATOL
#   ||G - G_ref||_F      <= GRAD_FRO_REL * ||G_ref||_F + GRAD_ATOL * sqrt(n)
# The kernel rounds P and dS to bf16 (unit roundoff u = 2^-8) before their
# products and writes bf16 outputs (another u per element); D = <dO, O> uses
# the bf16 forward output.  Emulating exactly those roundings on the CPU gives
# normwise errors of 2.3e-3 (N(0,1) inputs) to 4.8e-3 (Q, K ~ N(0, 3^2)) and
# worst elements at 6.7e-3 of max |G_ref|; the bounds are about 2x and 3x
# those, i.e. about 2.5u normwise and 5u elementwise.  GRAD_ATOL covers
# gradients that are exactly zero in fp64 (e.g. dQ, dK with one key) and come
# out as fp32 rounding noise.
GRAD_MAX_REL = 2e-2
GRAD_FRO_REL = 1e-2
GRAD_ATOL = 1e-4


def check_grad(g_gpu, g_ref, label=""):
    """Assert the gradient tolerances for one head's [rows, d] gradient;
    return (max err / max |ref|, normwise relative error)."""
    assert np.isfinite(g_gpu).all(), f"{label}: non-finite gradient"
    err = np.abs(g_gpu - g_ref)
    ref_max = float(np.abs(g_ref).max()) if g_ref.size else 0.0
    bound = GRAD_MAX_REL * ref_max + GRAD_ATOL
    assert err.max() <= bound, (f"{label}: max err {err.max():.3e} > {bound:.3e} "
                                f"(max |ref| {ref_max:.3e})")
    fro_ref = float(np.linalg.norm(g_ref))
    fro_err = float(np.linalg.norm(err))
    fbound = GRAD_FRO_REL * fro_ref + GRAD_ATOL * math.sqrt(err.size)
    assert fro_err <= fbound, f"{label}: normwise err {fro_err:.3e} > {fbound:.3e}"
    return (float(err.max()) / ref_max if ref_max else 0.0,
            fro_err / fro_ref if fro_ref else 0.0)


def check_grads_per_head(got, ref, label=""):
    """got/ref: (dq, dk, dv) arrays [..., L, d]; checks every head."""
    worst = {}
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        g = g.reshape(-1, g.shape[-2], g.shape[-1])
        r = r.reshape(-1, r.shape[-2], r.shape[-1])
        for h in range(g.shape[0]):
            m, f = check_grad(g[h], r[h], f"{label} {name} head {h}")
            worst[name] = max(worst.get(name, (0, 0))[0], m), max(worst.get(name, (0, 0))[1], f)
    return worst
