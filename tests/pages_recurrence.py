"""The pages' online-softmax recurrences in fp64, used to pin the oracle.

These are independent restatements of the METHOD (tiling + online softmax),
written from the pages' equations; the oracle states the plain definition.
The pages claim the two reach the same result exactly (up to rounding), so
agreement between them pins the oracle.  Test code only.
"""

from __future__ import annotations

import numpy as np


def online_sum_exp(x, block):
    """Blocked one-pass sum of exponentials.

    "大语言模型研究14——注意力机制优化之FlashAttention", section 1.1, eq. (4)-(7):
    m_k = max(m_{k-1}, max x_k);  s_k = e^{m_{k-1} - m_k} s_{k-1} + b_k with
    b_k = sum_{j in block k} e^{x_j - m_k}.  Returns (m_K, s_K) and the
    per-block history [(m_k, s_k)].
    """
    x = np.asarray(x, dtype=np.float64)
    m, s = -np.inf, 0.0
    hist = []
    for lo in range(0, x.size, block):
        xk = x[lo:lo + block]
        m_new = max(m, float(xk.max()))
        b = float(np.exp(xk - m_new).sum())
        s = (np.exp(m - m_new) if m != -np.inf else 0.0) * s + b
        m = m_new
        hist.append((m, s))
    return m, s, hist


def tiled_attention(q, k, v, scale, causal, block_r, block_c, trace=None):
    """FlashAttention-2 forward (one head) with online softmax, fp64.

    Follows "04 Transformers, Attention, and FlashAttention", Algorithm 1:
    Q in T_r blocks of B_r rows (step 1); per Q block, O = 0, l = 0,
    m = -inf (step 5); per K/V block: S = Q_i K_j^T (step 8, here with the
    scale applied to S as on "FlashAttention: как реально считается attention
    на GPU", section "Формулы online softmax"), m_new = max(m, rowmax S),
    P~ = exp(S - m_new), l = e^{m - m_new} l + rowsum P~ (step 9),
    O = diag(e^{m - m_new}) O + P~ V_j (step 10, multiplying by the
    correction as the step's prose and the other pages state), then O / l
    (step 12) and L = m + log l (step 13).  The causal mask keeps key <= query
    ("FlashAttention 深度解析", second part, section 2.3) and skips blocks that
    lie wholly above the diagonal.  A row whose running max is still -inf
    takes correction 0 (the guard printed on the page-3 toy).

    ``trace``, if a list, receives (i_block, j_block, m, l, O_unnormalised)
    after every K/V block, for the induction pin.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    L, d = q.shape
    out = np.zeros((L, d))
    lse = np.zeros(L)
    for i0 in range(0, L, block_r):
        qi = q[i0:i0 + block_r]
        rows = np.arange(i0, i0 + qi.shape[0])
        m = np.full(qi.shape[0], -np.inf)
        l = np.zeros(qi.shape[0])
        o = np.zeros((qi.shape[0], d))
        for j0 in range(0, L, block_c):
            if causal and j0 > rows[-1]:
                break  # every key of this block lies after every query of the tile
            kj = k[j0:j0 + block_c]
            vj = v[j0:j0 + block_c]
            s = scale * (qi @ kj.T)
            if causal:
                cols = np.arange(j0, j0 + kj.shape[0])
                s = np.where(cols[None, :] <= rows[:, None], s, -np.inf)
            m_new = np.maximum(m, s.max(axis=1))
            ref = np.where(np.isneginf(m_new), 0.0, m_new)
            p = np.exp(s - ref[:, None])
            corr = np.where(np.isneginf(m), 0.0, np.exp(m - ref))
            l = corr * l + p.sum(axis=1)
            o = corr[:, None] * o + p @ vj
            m = m_new
            if trace is not None:
                trace.append((i0 // block_r, j0 // block_c, m.copy(), l.copy(), o.copy()))
        out[i0:i0 + qi.shape[0]] = o / l[:, None]
        lse[i0:i0 + qi.shape[0]] = m + np.log(l)
    return out, lse
