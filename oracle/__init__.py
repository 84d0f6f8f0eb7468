"""fp64 CPU oracle for the attention forward pass and its gradients.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``; never by the product package.
It shares no code with the CUDA path; the two meet only in the seeded input
generator (:mod:`fa_inputs`), which holds no attention arithmetic.

Two statements of the same plain definition (three-step attention,
"FlashAttention 深度解析", first part, section 2.3; log-sum-exp per row,
"04 Transformers, Attention, and FlashAttention", Algorithm 1, steps 13-15):

* :func:`attention` -- the C implementation (``attention_fp64.c``), row by
  row, threaded; used at every size.
* :func:`attention_numpy` -- the same definition in matrix form with numpy
  (a library matmul per product), for small cases.

Gradients (the backward pass by recomputation, "FlashAttention 深度解析",
first part, sections 4.1-4.2; chain rule through the scaled scores):

* :func:`attention_bwd` -- C implementation (``attention_bwd_fp64.c``) in
  three passes (row statistics, per-key dK/dV, per-query dQ), threaded,
  optionally restricted to chosen rows so that rows of large problems are
  affordable.
* :func:`attention_bwd_numpy` -- the same formulas in matrix form.

FP8: :mod:`oracle.fp8` holds the E4M3 block quantisation of Q and K
("FlashAttention 深度解析", third part, section 2.3); the FP8 forward's
expected result is :func:`attention` on the de-quantised inputs.

Parity status: pinned (forward, gradients, FP8 quantisation).  The pins (``tests/test_oracle_pins.py``) check both
against the worked example printed on "FlashAttention: как реально
считается attention на GPU" (section "Код: от игрушечного NumPy до реального
PyTorch"), against high-precision brute force, closed forms and invariants.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

__all__ = ["attention", "attention_numpy", "attention_bf16", "row_probs", "attention_bwd",
           "attention_bwd_numpy", "lib"]

_lib = None


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int64)
        L.oracle_attention_fp64.argtypes = [dp, dp, dp, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_double, ctypes.c_int,
                                            ip, ctypes.c_int64, dp, dp, ctypes.c_int]
        L.oracle_attention_fp64.restype = ctypes.c_int
        L.oracle_row_probs_fp64.argtypes = [dp, dp, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_double, ctypes.c_int, ctypes.c_int64, dp]
        L.oracle_row_probs_fp64.restype = ctypes.c_int
        L.oracle_attention_bwd_fp64.argtypes = [dp, dp, dp, dp, ctypes.c_int64, ctypes.c_int64,
                                                ctypes.c_int64, ctypes.c_double, ctypes.c_int,
                                                ip, ctypes.c_int64, ip, ctypes.c_int64,
                                                dp, dp, dp, ctypes.c_int]
        L.oracle_attention_bwd_fp64.restype = ctypes.c_int
        _lib = L
    return _lib


def _dptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def attention(q, k, v, scale, causal=False, rows=None, threads=0):
    """Exact attention in fp64 (C implementation).

    q, k, v: float64 arrays [..., L, d] (leading dims are heads, flattened).
    rows: optional flat query indices (head * L + i); default every row.
    Returns (o, lse): o [n_rows, d] (or q's shape when rows is None) and
    lse [n_rows] (or q's shape without d).
    """
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    if q.shape != k.shape or q.shape != v.shape or q.ndim < 2:
        raise ValueError("q, k, v must share one shape [..., L, d]")
    L, d = q.shape[-2], q.shape[-1]
    n_heads = int(np.prod(q.shape[:-2], dtype=np.int64)) if q.ndim > 2 else 1
    if rows is None:
        n_rows = n_heads * L
        rows_arr = None
        rp = ctypes.POINTER(ctypes.c_int64)()
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64).ravel()
        n_rows = rows_arr.size
        rp = rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    o = np.empty((n_rows, d), dtype=np.float64)
    lse = np.empty(n_rows, dtype=np.float64)
    rc = lib().oracle_attention_fp64(_dptr(q), _dptr(k), _dptr(v), n_heads, L, d,
                                     float(scale), int(bool(causal)), rp, n_rows,
                                     _dptr(o), _dptr(lse), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_fp64 failed with code {rc}")
    if rows is None:
        return o.reshape(q.shape), lse.reshape(q.shape[:-1])
    return o, lse


def attention_bf16(q_bits, k_bits, v_bits, scale, causal=False, rows=None, threads=0):
    """:func:`attention` on bfloat16 bit patterns (uint16), promoted exactly."""
    from fa_inputs import bf16_bits_to_float32
    f = lambda b: bf16_bits_to_float32(b).astype(np.float64)
    return attention(f(q_bits), f(k_bits), f(v_bits), scale, causal, rows, threads)


def row_probs(q, k, scale, causal, i):
    """Softmax probabilities of query row ``i`` of one head (C implementation)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    L, d = q.shape
    p = np.empty(L, dtype=np.float64)
    rc = lib().oracle_row_probs_fp64(_dptr(q), _dptr(k), L, d, float(scale),
                                     int(bool(causal)), int(i), _dptr(p))
    if rc != 0:
        raise RuntimeError(f"oracle_row_probs_fp64 failed with code {rc}")
    return p


def attention_numpy(q, k, v, scale, causal=False):
    """The same definition in matrix form (numpy fp64), for small cases.

    S = scale * Q K^T; masked scores (key > query when causal) are removed
    by -inf; P = exp(S - rowmax) / rowsum; O = P V; lse = rowmax + log rowsum.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    L = q.shape[-2]
    s = scale * np.matmul(q, np.swapaxes(k, -1, -2))
    if causal:
        allowed = np.tril(np.ones((L, L), dtype=bool))
        s = np.where(allowed, s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    z = e.sum(axis=-1, keepdims=True)
    o = np.matmul(e / z, v)
    lse = (m + np.log(z))[..., 0]
    return o, lse


def _rows_arg(rows, n_flat):
    if rows is None:
        return None, n_flat, ctypes.POINTER(ctypes.c_int64)()
    arr = np.ascontiguousarray(rows, dtype=np.int64).ravel()
    return arr, arr.size, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def attention_bwd(q, k, v, dout, scale, causal=False, key_rows=None, query_rows=None,
                  threads=0):
    """Gradients dQ, dK, dV of exact attention in fp64 (C implementation).

    q, k, v, dout: float64 arrays [..., L, d] (leading dims are heads).
    key_rows / query_rows: optional flat indices (head * L + row) of the
    dK/dV rows and the dQ rows wanted; default every row.  An empty list
    skips that gradient.
    Returns (dq, dk, dv): each shaped like q when its rows are all wanted,
    else [n_rows, d].
    """
    q, k, v, dout = (np.ascontiguousarray(a, dtype=np.float64) for a in (q, k, v, dout))
    if not (q.shape == k.shape == v.shape == dout.shape) or q.ndim < 2:
        raise ValueError("q, k, v, dout must share one shape [..., L, d]")
    L, d = q.shape[-2], q.shape[-1]
    n_heads = int(np.prod(q.shape[:-2], dtype=np.int64)) if q.ndim > 2 else 1
    n_flat = n_heads * L
    karr, nk, kp = _rows_arg(key_rows, n_flat)
    qarr, nq, qp = _rows_arg(query_rows, n_flat)
    dq = np.empty((nq, d), dtype=np.float64)
    dk = np.empty((nk, d), dtype=np.float64)
    dv = np.empty((nk, d), dtype=np.float64)
    rc = lib().oracle_attention_bwd_fp64(_dptr(q), _dptr(k), _dptr(v), _dptr(dout), n_heads,
                                         L, d, float(scale), int(bool(causal)), kp, nk, qp,
                                         nq, _dptr(dq), _dptr(dk), _dptr(dv), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_bwd_fp64 failed with code {rc}")
    if query_rows is None:
        dq = dq.reshape(q.shape)
    if key_rows is None:
        dk, dv = dk.reshape(q.shape), dv.reshape(q.shape)
    return dq, dk, dv


def attention_bwd_numpy(q, k, v, dout, scale, causal=False):
    """The same gradients in matrix form (numpy fp64), for small cases.

    P = softmax(scale * Q K^T) (masked entries 0); dV = P^T dO; dP = dO V^T;
    dS = P * (dP - rowsum(dP * P)); dQ = scale * dS K; dK = scale * dS^T Q.
    """
    q, k, v, dout = (np.asarray(a, dtype=np.float64) for a in (q, k, v, dout))
    L = q.shape[-2]
    s = scale * np.matmul(q, np.swapaxes(k, -1, -2))
    if causal:
        s = np.where(np.tril(np.ones((L, L), dtype=bool)), s, -np.inf)
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    p = e / e.sum(axis=-1, keepdims=True)
    dv = np.matmul(np.swapaxes(p, -1, -2), dout)
    dp = np.matmul(dout, np.swapaxes(v, -1, -2))
    ds = p * (dp - (dp * p).sum(axis=-1, keepdims=True))
    dq = scale * np.matmul(ds, k)
    dk = scale * np.matmul(np.swapaxes(ds, -1, -2), q)
    return dq, dk, dv
