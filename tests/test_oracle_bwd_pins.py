"""Pins for the fp64 gradient oracle: checks that do not restate its formulas.

The gradients are pinned to the forward definition itself, by central
finite differences of the scalar <dO, O(Q, K, V)> computed with the
(separately pinned) forward oracle, and to identities that any correct
gradient of softmax attention satisfies:

* sum_j dK_j = 0: every row of dS sums to zero (softmax is invariant to a
  shift of its scores), so dK = scale * dS^T Q sums to zero over the keys;
* sum_j dV_j = sum_i dO_i: every row of P sums to one;
* linearity in dO;
* one key (L = 1): P = 1, so dV = dO and dQ = dK = 0;
* equal keys: the scores of a row are all equal, so dQ = 0;
* the row sum of the backward formula equals dO_i . O_i (the identity
  FlashAttention-2 kernels use for it; here it checks the oracle's row sum
  against the forward output);
* causal: query 0 sees one key (dQ_0 = 0), and key L-1 is seen only by
  query L-1 (dV_{L-1} = P_{L-1,L-1} dO_{L-1}, with that probability from the
  forward oracle).

Everything runs on the CPU.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle


def _loss(q, k, v, dout, scale, causal):
    o, _ = oracle.attention(q, k, v, scale, causal)
    return float(np.sum(dout * o))


def finite_difference_grads(q, k, v, dout, scale, causal, h=1e-5):
    """Central differences of <dO, O> with respect to every input element."""
    grads = []
    args = [q.copy(), k.copy(), v.copy()]
    for which in range(3):
        g = np.zeros_like(args[which])
        flat = args[which].reshape(-1)
        for e in range(flat.size):
            keep = flat[e]
            flat[e] = keep + h
            up = _loss(*args, dout, scale, causal)
            flat[e] = keep - h
            down = _loss(*args, dout, scale, causal)
            flat[e] = keep
            g.reshape(-1)[e] = (up - down) / (2 * h)
        grads.append(g)
    return grads


def _inputs(heads, L, d, seed, std=1.0):
    rng = np.random.default_rng(seed)
    return [rng.normal(0.0, std, size=(heads, L, d)) for _ in range(3)] + \
           [rng.normal(0.0, 1.0, size=(heads, L, d))]


def pins_pass(bwd) -> bool:
    """Every pin below, applied to a candidate gradient function
    bwd(q, k, v, dout, scale, causal) -> (dq, dk, dv)."""
    for causal in (False, True):
        q, k, v, do = _inputs(2, 6, 3, 11 + causal, 1.3)
        fd = finite_difference_grads(q, k, v, do, 0.8, causal)
        got = bwd(q, k, v, do, 0.8, causal)
        for a, b in zip(got, fd):
            if np.abs(a - b).max() > 1e-7:
                return False
        q, k, v, do = _inputs(2, 40, 8, 21 + causal)
        dq, dk, dv = bwd(q, k, v, do, 0.5, causal)
        if np.abs(dk.sum(axis=1)).max() > 1e-12:
            return False
        if np.abs(dv.sum(axis=1) - do.sum(axis=1)).max() > 1e-12:
            return False
        if causal:
            if np.abs(dq[:, 0]).max() > 1e-15:
                return False
            for h in range(q.shape[0]):
                p_last = oracle.row_probs(q[h], k[h], 0.5, True, q.shape[1] - 1)[-1]
                if np.abs(dv[h, -1] - p_last * do[h, -1]).max() > 1e-14:
                    return False
    return True


def test_oracle_passes_the_pins():
    assert pins_pass(lambda *a: oracle.attention_bwd(*a))
    assert pins_pass(lambda *a: oracle.attention_bwd_numpy(*a))


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences_wider(causal):
    # larger spread of scores (peaked softmax rows) and a negative scale
    q, k, v, do = _inputs(1, 9, 5, 31 + causal, 2.5)
    fd = finite_difference_grads(q, k, v, do, -0.7, causal)
    got = oracle.attention_bwd(q, k, v, do, -0.7, causal)
    for name, a, b in zip(("dq", "dk", "dv"), got, fd):
        assert np.abs(a - b).max() <= 1e-7 * max(1.0, np.abs(b).max()), name


@pytest.mark.parametrize("causal", [False, True])
def test_linear_in_output_gradient(causal):
    q, k, v, d1 = _inputs(2, 33, 16, 41 + causal)
    d2 = np.random.default_rng(7).normal(size=d1.shape)
    a = oracle.attention_bwd(q, k, v, d1, 0.3, causal)
    b = oracle.attention_bwd(q, k, v, d2, 0.3, causal)
    c = oracle.attention_bwd(q, k, v, 2.0 * d1 - 3.0 * d2, 0.3, causal)
    for x, y, z in zip(a, b, c):
        assert np.abs(z - (2.0 * x - 3.0 * y)).max() <= 1e-12


def test_single_key():
    q, k, v, do = _inputs(3, 1, 8, 51)
    for causal in (False, True):
        dq, dk, dv = oracle.attention_bwd(q, k, v, do, 0.9, causal)
        assert np.array_equal(dv, do)
        assert np.abs(dq).max() == 0.0 and np.abs(dk).max() == 0.0


def test_equal_keys_give_zero_dq():
    q, k, v, do = _inputs(1, 24, 8, 61)
    k[:] = k[:, :1, :]
    for causal in (False, True):
        dq, _, _ = oracle.attention_bwd(q, k, v, do, 0.7, causal)
        assert np.abs(dq).max() <= 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_row_sum_equals_do_dot_o(causal):
    # rowsum(dP * P)_i = sum_j P_ij <dO_i, v_j> = <dO_i, O_i>.  With every key
    # equal to the ones vector, dQ_i = scale * sum_j dS_ij, which is zero only
    # if the oracle subtracts exactly that row sum.
    q, k, v, do = _inputs(1, 30, 8, 71 + causal)
    o, _ = oracle.attention(q, k, v, 0.6, causal)
    probe_k = np.ones_like(k)
    dq, _, _ = oracle.attention_bwd(q, probe_k, v, do, 0.6, causal)
    assert np.abs(dq).max() <= 1e-13
    # and the row sum itself, from the matrix form, equals <dO_i, O_i>
    s = 0.6 * q[0] @ k[0].T
    if causal:
        s = np.where(np.tril(np.ones((30, 30), bool)), s, -np.inf)
    p = np.exp(s - s.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    rowsum = ((do[0] @ v[0].T) * p).sum(1)
    assert np.abs(rowsum - (do[0] * o[0]).sum(1)).max() <= 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_chosen_rows_equal_full(causal):
    q, k, v, do = _inputs(3, 50, 8, 81 + causal)
    full = oracle.attention_bwd(q, k, v, do, 0.4, causal)
    keys = [0, 49, 77, 149]
    queries = [3, 50, 149]
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, 0.4, causal, key_rows=keys, query_rows=queries)
    assert np.array_equal(dq, full[0].reshape(-1, 8)[queries])
    assert np.array_equal(dk, full[1].reshape(-1, 8)[keys])
    assert np.array_equal(dv, full[2].reshape(-1, 8)[keys])
    # an empty list skips that gradient
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, 0.4, causal, key_rows=[], query_rows=[5])
    assert dk.shape == (0, 8) and dv.shape == (0, 8)
    assert np.array_equal(dq[0], full[0].reshape(-1, 8)[5])


def test_thread_count_does_not_change_bits():
    q, k, v, do = _inputs(2, 64, 16, 91)
    a = oracle.attention_bwd(q, k, v, do, 0.25, True, threads=1)
    b = oracle.attention_bwd(q, k, v, do, 0.25, True, threads=7)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_rejects_bad_arguments():
    q, k, v, do = _inputs(1, 8, 4, 3)
    with pytest.raises(RuntimeError):
        oracle.attention_bwd(q, k, v, do, 0.5, False, key_rows=[8])
    with pytest.raises(ValueError):
        oracle.attention_bwd(q, k, v, do[:, :4], 0.5, False)
