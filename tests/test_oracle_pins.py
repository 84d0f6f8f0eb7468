"""Pins for the fp64 oracle: checks against what the pages and mathematics fix.

Every test here runs on the CPU.  None compares the oracle with itself:
each pin is a worked example from the pages, a closed form, an invariant,
an independent high-precision brute force, or the pages' own tiled
recurrence (a different algorithm that the pages prove reaches the same
result).
"""

from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest

import oracle
from fa_inputs import bf16_bits_to_float32, make_custom
from tests.pages_recurrence import online_sum_exp, tiled_attention

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_normals(shape, seed, std=1.0):
    q, k, v = make_custom(1, 1, shape[0], shape[1], seed, std, std, 1.0)
    f = lambda b: bf16_bits_to_float32(b).astype(np.float64)[0, 0]
    return f(q), f(k), f(v)


# --------------------------------------------------------------------------
# P1. The NumPy toy printed on the page-3 article: tiled == naive in fp64.
# --------------------------------------------------------------------------
def test_page3_numpy_toy_golden():
    g = json.load(open(os.path.join(GOLDEN, "page3_numpy_toy.json")))
    rs = np.random.RandomState(42)
    Q = rs.standard_normal((g["N"], g["D"]))
    K = rs.standard_normal((g["N"], g["D"]))
    V = rs.standard_normal((g["N"], g["D"]))
    scale = 1.0 / math.sqrt(g["D"])
    o_c, lse_c = oracle.attention(Q, K, V, scale)
    o_np, _ = oracle.attention_numpy(Q, K, V, scale)
    o_t, lse_t = tiled_attention(Q, K, V, scale, False, g["N"], g["BLOCK"])
    # the page's assertion (atol 1e-10) and its printed size (a few ulp)
    assert np.allclose(o_c, o_t, rtol=0, atol=g["page_assert_atol"])
    assert np.abs(o_c - o_t).max() <= 8 * g["printed_max_abs_diff"]
    assert np.abs(o_np - o_t).max() <= 8 * g["printed_max_abs_diff"]
    assert np.abs(lse_c - lse_t).max() <= 1e-14


# --------------------------------------------------------------------------
# P2. One-row walk-through (page 3): 4 blocks of 4 keys; correction 1.0 at
#     the last block; result == one-shot softmax over the 16 scores.
# --------------------------------------------------------------------------
def test_page3_one_row_walkthrough():
    g = json.load(open(os.path.join(GOLDEN, "page3_walkthrough.json")))
    nb, bs = g["n_blocks"], g["keys_per_block"]
    n = nb * bs
    d = 8
    rng = np.random.default_rng(7)
    # scores chosen so that the running max grows in blocks 1..3, not in 4
    target = np.concatenate([rng.uniform(-1, 0, bs), rng.uniform(0, 1, bs),
                             rng.uniform(1, 2, bs), rng.uniform(-2, 1, bs)])
    q = np.zeros((1, d)); q[0, 0] = 1.0
    k = np.zeros((n, d)); k[:, 0] = target
    v = rng.standard_normal((n, d))
    m, l, o = -np.inf, 0.0, np.zeros(d)
    corrections = []
    for b in range(nb):
        s = target[b * bs:(b + 1) * bs]
        m_new = max(m, s.max())
        c = 0.0 if m == -np.inf else math.exp(m - m_new)
        p = np.exp(s - m_new)
        l = c * l + p.sum()
        o = c * o + p @ v[b * bs:(b + 1) * bs]
        m = m_new
        corrections.append(c)
    assert corrections[-1] == g["correction_at_last_block"]
    assert all(c < 1.0 for c in corrections[1:-1])
    # the oracle for query row 0 against the 16 keys (pad q to L rows)
    qq = np.zeros((n, d)); qq[0] = q[0]
    o_or, lse_or = oracle.attention(qq, k, v, 1.0, rows=[0])
    assert np.abs(o_or[0] - o / l).max() <= 1e-14
    assert abs(lse_or[0] - (m + math.log(l))) <= 1e-14
    p_or = oracle.row_probs(qq, k, 1.0, False, 0)
    assert np.abs(p_or @ v - o / l).max() <= 1e-14


# --------------------------------------------------------------------------
# P3. Page-4 recurrence s_k = e^{m_{k-1}-m_k} s_{k-1} + b_k == two-pass sum.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n", [1, 2, 5, 16, 17, 64, 1000])
@pytest.mark.parametrize("block", [1, 3, 4, 16])
def test_recurrence_equals_two_pass(n, block):
    rng = np.random.default_rng(1000 * n + block)
    x = rng.normal(0.0, 5.0, n)
    m, s, _ = online_sum_exp(x, block)
    two_pass_m = x.max()
    two_pass_s = np.exp(x - two_pass_m).sum()
    assert m == two_pass_m
    assert abs(s - two_pass_s) <= 1e-12 * two_pass_s
    # and the oracle's LSE of a one-row problem with these scores
    d = 2
    q = np.zeros((n, d)); q[:, 0] = 1.0
    k = np.zeros((n, d)); k[:, 0] = x
    v = np.ones((n, d))
    _, lse = oracle.attention(q, k, v, 1.0, rows=[0])
    assert abs(lse[0] - (m + math.log(s))) <= 1e-12 * max(1.0, abs(lse[0]))


# --------------------------------------------------------------------------
# P4. Induction invariant (page 1, section 3.4): after K/V block j the tiled
#     state equals exact attention over the keys seen so far.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_induction_invariant_against_prefix_oracle(causal):
    L, d, br, bc = 40, 8, 16, 8
    q, k, v = _bf16_normals((L, d), 11)
    scale = 1.0 / math.sqrt(d)
    trace = []
    tiled_attention(q, k, v, scale, causal, br, bc, trace)
    for ib, jb, m, l, o in trace:
        end = min(L, (jb + 1) * bc)
        rows = np.arange(ib * br, min(L, (ib + 1) * br))
        kp, vp = k[:end], v[:end]
        qp = np.zeros((end, d))
        # exact attention of these query rows over the key prefix [0, end)
        for t, r in enumerate(rows):
            qp[0] = q[r]
            n_keys = min(end, r + 1) if causal else end
            o_ex, lse_ex = oracle.attention(qp[:n_keys], kp[:n_keys], vp[:n_keys], scale, rows=[0])
            assert abs((m[t] + math.log(l[t])) - lse_ex[0]) <= 1e-12
            assert np.abs(o[t] / l[t] - o_ex[0]).max() <= 1e-12


# --------------------------------------------------------------------------
# P5. Invariants and closed forms.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_softmax_rows_sum_to_one(causal):
    q, k, _ = _bf16_normals((64, 16), 3, std=3.0)
    for i in (0, 1, 31, 63):
        p = oracle.row_probs(q, k, 0.25, causal, i)
        assert abs(p.sum() - 1.0) <= 1e-12
        assert (p >= 0).all()
        if causal:
            assert (p[i + 1:] == 0).all() and (p[:i + 1] > 0).all()


@pytest.mark.parametrize("causal", [False, True])
def test_identical_value_rows(causal):
    q, k, _ = _bf16_normals((50, 16), 4)
    row = np.linspace(-2, 2, 16)
    v = np.tile(row, (50, 1))
    o, _ = oracle.attention(q, k, v, 0.3, causal)
    assert np.abs(o - row).max() <= 1e-14


def test_causal_first_row_is_v0_exactly():
    q, k, v = _bf16_normals((33, 64), 5)
    scale = 0.125
    o, lse = oracle.attention(q, k, v, scale, True)
    assert np.array_equal(o[0], v[0])
    assert lse[0] == scale * float(np.dot(q[0], k[0]))


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_is_mean_and_log_count(causal):
    L, d = 37, 8
    q, k, v = _bf16_normals((L, d), 6)
    o, lse = oracle.attention(q, k, v, 0.0, causal)
    for i in range(L):
        n = i + 1 if causal else L
        assert np.abs(o[i] - v[:n].mean(axis=0)).max() <= 1e-14
        assert abs(lse[i] - math.log(n)) <= 1e-14


def test_permuting_keys_with_values_non_causal():
    q, k, v = _bf16_normals((48, 16), 8)
    perm = np.random.default_rng(0).permutation(48)
    o1, l1 = oracle.attention(q, k, v, 0.25)
    o2, l2 = oracle.attention(q, k[perm], v[perm], 0.25)
    assert np.abs(o1 - o2).max() <= 1e-13
    assert np.abs(l1 - l2).max() <= 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_value_shift(causal):
    q, k, v = _bf16_normals((30, 8), 9)
    o1, _ = oracle.attention(q, k, v, 0.5, causal)
    o2, _ = oracle.attention(q, k, v + 1.5, 0.5, causal)
    assert np.abs((o2 - o1) - 1.5).max() <= 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_lse_bounds_and_logsumexp(causal):
    from scipy.special import logsumexp
    L, d, scale = 64, 32, 1.0 / math.sqrt(32)
    q, k, v = _bf16_normals((L, d), 10, std=3.0)
    _, lse = oracle.attention(q, k, v, scale, causal)
    s_full = scale * (q @ k.T)
    for i in range(L):
        n = i + 1 if causal else L
        s = s_full[i, :n]
        assert s.max() <= lse[i] + 1e-12
        assert lse[i] <= s.max() + math.log(n) + 1e-12
        assert abs(lse[i] - logsumexp(s)) <= 1e-12 * max(1.0, abs(lse[i]))


def test_large_logits_do_not_overflow():
    # scores around 1e3 would overflow exp() without the max subtraction
    L, d = 16, 4
    q = np.zeros((L, d)); q[:, 0] = 40.0
    k = np.zeros((L, d)); k[:, 0] = np.arange(L)
    v = np.eye(L, d)
    o, lse = oracle.attention(q, k, v, 2.0)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    # the last key dominates completely (gap 80 in the exponent)
    assert abs(lse[0] - 2.0 * 40.0 * (L - 1)) <= 1e-9


# --------------------------------------------------------------------------
# P6. Brute force, L <= 16: exact products, 60-digit exponentials, no max
#     subtraction (an independent route to the same numbers).
# --------------------------------------------------------------------------
def _brute(q, k, v, scale, causal):
    mpmath = pytest.importorskip("mpmath")
    from fractions import Fraction
    mpmath.mp.dps = 60
    L, d = q.shape
    o = np.zeros((L, d)); lse = np.zeros(L)
    sc = mpmath.mpf(Fraction(scale).numerator) / mpmath.mpf(Fraction(scale).denominator)
    for i in range(L):
        n = i + 1 if causal else L
        w = []
        for j in range(n):
            dot = sum(Fraction(float(q[i, t])) * Fraction(float(k[j, t])) for t in range(d))
            w.append(mpmath.exp(sc * mpmath.mpf(dot.numerator) / dot.denominator))
        z = mpmath.fsum(w)
        for t in range(d):
            o[i, t] = float(mpmath.fsum(w[j] * mpmath.mpf(float(v[j, t])) for j in range(n)) / z)
        lse[i] = float(mpmath.log(z))
    return o, lse


@pytest.mark.parametrize("L", [1, 2, 5, 16])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("scale", [0.125, 1.0])
def test_brute_force_small(L, causal, scale):
    d = 8
    q, k, v = _bf16_normals((L, d), 100 + L)
    o_b, lse_b = _brute(q, k, v, scale, causal)
    for o, lse in (oracle.attention(q, k, v, scale, causal),
                   oracle.attention_numpy(q, k, v, scale, causal)):
        assert np.abs(o - o_b).max() <= 1e-13
        assert np.abs(lse - lse_b).max() <= 1e-13


def test_brute_force_asymmetric_operands():
    # Q != K with a skewed pattern: a transposed product S^T would differ.
    L, d = 6, 3
    q = np.arange(L * d, dtype=np.float64).reshape(L, d) / 8.0
    k = (np.arange(L * d, dtype=np.float64).reshape(L, d)[::-1] - 4.0) / 16.0
    v = np.arange(L * d, dtype=np.float64).reshape(L, d) % 5
    o_b, lse_b = _brute(q, k, v, 0.5, False)
    o, lse = oracle.attention(q, k, v, 0.5)
    assert np.abs(o - o_b).max() <= 1e-13 and np.abs(lse - lse_b).max() <= 1e-13


# --------------------------------------------------------------------------
# P6b. Tiled recurrence vs oracle at every block size 1..L.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_tiled_every_block_size(causal):
    L, d = 13, 4
    q, k, v = _bf16_normals((L, d), 12, std=2.0)
    o_or, lse_or = oracle.attention(q, k, v, 0.7, causal)
    for br in (1, 4, L):
        for bc in range(1, L + 1):
            o_t, lse_t = tiled_attention(q, k, v, 0.7, causal, br, bc)
            assert np.abs(o_t - o_or).max() <= 1e-13
            assert np.abs(lse_t - lse_or).max() <= 1e-13


# --------------------------------------------------------------------------
# P7. The page-1 equivalence tests, redone in fp64 (B=2, H=4, L=128, d=64,
#     blocks of 32; causal with blocks of 64).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal,block", [(False, 32), (True, 64)])
def test_page1_equivalence_fp64(causal, block):
    B, H, L, d = 2, 4, 128, 64
    qb, kb, vb = make_custom(B, H, L, d, 42)
    f = lambda b: bf16_bits_to_float32(b).astype(np.float64)
    q, k, v = f(qb), f(kb), f(vb)
    scale = 1.0 / math.sqrt(d)
    o_or, lse_or = oracle.attention(q, k, v, scale, causal)
    for b in range(B):
        for h in range(H):
            o_t, lse_t = tiled_attention(q[b, h], k[b, h], v[b, h], scale, causal, block, block)
            assert np.abs(o_t - o_or[b, h]).max() <= 1e-12
            assert np.abs(lse_t - lse_or[b, h]).max() <= 1e-12


def test_c_and_numpy_statements_agree_and_threads_do_not_matter():
    qb, kb, vb = make_custom(2, 3, 70, 16, 5)
    f = lambda b: bf16_bits_to_float32(b).astype(np.float64)
    q, k, v = f(qb), f(kb), f(vb)
    for causal in (False, True):
        o1, l1 = oracle.attention(q, k, v, 0.25, causal, threads=1)
        o4, l4 = oracle.attention(q, k, v, 0.25, causal, threads=4)
        assert np.array_equal(o1, o4) and np.array_equal(l1, l4)
        o2, l2 = oracle.attention_numpy(q, k, v, 0.25, causal)
        assert np.abs(o1 - o2).max() <= 1e-13 and np.abs(l1 - l2).max() <= 1e-13
        rows = np.array([0, 69, 70, 139, 3 * 70 + 5])
        o_r, l_r = oracle.attention(q, k, v, 0.25, causal, rows=rows)
        assert np.array_equal(o_r, o1.reshape(-1, 16)[rows])
        assert np.array_equal(l_r, l1.reshape(-1)[rows])


def test_oracle_rejects_bad_arguments():
    q = np.zeros((4, 2))
    with pytest.raises(RuntimeError):
        oracle.attention(q, q, q, 1.0, rows=[4 * 1 + 7])
    with pytest.raises(ValueError):
        oracle.attention(q, q[:3], q, 1.0)


# --------------------------------------------------------------------------
# P8. Flash-Decoding ("04 Transformers, Attention, and FlashAttention",
#     Flash-Decoding): attention over key chunks, merged by their log-sum-exp
#     weights, equals attention over all keys.  Pins the merge rule the
#     split-KV path uses, with the oracle on each chunk.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("cuts", [(25,), (1, 49), (10, 20, 30, 40), (49,)])
def test_split_and_merge_equals_whole(cuts):
    L, d = 50, 8
    q, k, v = _bf16_normals((L, d), 21, std=2.0)
    o_all, lse_all = oracle.attention(q, k, v, 0.5)
    bounds = [0, *cuts, L]
    # each chunk: every query against keys [lo, hi) only (non-causal, so the
    # oracle's matrix statement takes a key block of its own length)
    parts = [oracle.attention_numpy(q, k[lo:hi], v[lo:hi], 0.5)
             for lo, hi in zip(bounds[:-1], bounds[1:])]
    lses = np.stack([p[1] for p in parts])
    M = lses.max(axis=0)
    lse = M + np.log(np.exp(lses - M).sum(axis=0))
    o = sum(np.exp(p[1] - lse)[:, None] * p[0] for p in parts)
    assert np.abs(lse - lse_all).max() <= 1e-12
    assert np.abs(o - o_all).max() <= 1e-12
    # an empty chunk (log-sum-exp -inf) has weight exp(-inf - lse) = 0
    assert np.exp(-np.inf - lse).max() == 0.0
