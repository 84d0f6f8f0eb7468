"""FP8 (E4M3) block quantisation for the FP8 forward: the oracle's side.

TEST INFRASTRUCTURE ONLY (imported by ``tests/`` and the benchmark's CPU
legs, never by the product package).  It shares no code with the CUDA path.

What it follows.  "FlashAttention 深度解析", third part, section 2.3 (FP8 与
块量化): Q and K are split into blocks; each block gets the scale
s = max(|block|) / FP8_MAX and is stored as Quantize(block / s) in the E4M3
format; after the product the scores are de-quantised,
S = (Q_FP8 K_FP8^T) * s_q * s_k (times the softmax scale).  A block here is
128 consecutive rows of one head (the kernel's tile), all d columns.

E4M3 (the format, not a library): 1 sign bit, 4 exponent bits with bias 7,
3 mantissa bits; no infinities; exponent field 0 holds the subnormals
m * 2^-9 (m = 1..7); the largest finite value is 1.75 * 2^8 = 448; the code
with all exponent and mantissa bits set is NaN.  Quantize rounds to the
nearest representable value, ties to the even mantissa, and saturates
values beyond 448 to +-448.

Where floating point decides an integer (the code), the decision is taken
in the kernel's precision: the scale is the fp32 quotient amax / 448 and
the quantised argument the fp32 quotient x / s, both correctly rounded.
A block whose entries are all zero gets the scale 1 (its codes are 0).

Parity status: pinned (tests/test_oracle_fp8.py).
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
BLOCK_ROWS = 128


def e4m3_decode(codes) -> np.ndarray:
    """Codes (uint8) -> values (float64); NaN codes give NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 0xF) & (m == 0x7), np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """Values -> E4M3 codes: round to nearest, ties to even, saturate at
    +-448; NaN -> 0x7F.  Works on float64 views of the (fp32) inputs."""
    x = np.asarray(x, dtype=np.float64)
    nan = np.isnan(x)
    sign = np.signbit(x) & ~nan
    a = np.where(nan, 0.0, np.abs(x))
    # exponent of the binade (subnormal range uses the minimum exponent -6)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    quantum = np.exp2(e - 3.0)                   # spacing inside the binade
    q = a / quantum                               # exact: power-of-two division
    n = np.floor(q)
    frac = q - n
    n = n + ((frac > 0.5) | ((frac == 0.5) & (np.mod(n, 2) == 1)))
    r = n * quantum                               # rounded magnitude
    r = np.minimum(r, E4M3_MAX)                   # saturate
    # encode r
    with np.errstate(divide="ignore"):
        er = np.floor(np.log2(np.where(r > 0, r, 1.0)))
    sub = r < 2.0 ** -6
    m_sub = np.round(r / 2.0 ** -9)               # exact integers 0..7
    m_norm = np.round((r / np.exp2(er) - 1.0) * 8.0)
    code = np.where(sub, m_sub, (er + 7.0) * 8.0 + m_norm).astype(np.uint8)
    # the sign bit follows the input's sign bit (so -0 and negative values
    # that round to zero give 0x80, as an IEEE-style conversion does)
    code = np.where(sign, code | np.uint8(0x80), code).astype(np.uint8)
    return np.where(nan, np.uint8(0x7F), code).astype(np.uint8)


def block_scales(x, block_rows=BLOCK_ROWS) -> np.ndarray:
    """Per-block scales s = amax / 448 (fp32 division), amax over each block
    of ``block_rows`` rows of each head.  x: [heads, L, d] finite values
    representable in fp32 (the bf16 inputs)."""
    x = np.asarray(x, dtype=np.float32)
    H, L, _ = x.shape
    nb = (L + block_rows - 1) // block_rows
    s = np.empty((H, nb), dtype=np.float32)
    for b in range(nb):
        amax = np.abs(x[:, b * block_rows:(b + 1) * block_rows, :]).max(axis=(1, 2))
        s[:, b] = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0))
    return s


def quantize_blocks(x, block_rows=BLOCK_ROWS):
    """Block quantisation: (codes uint8 [heads, L, d], scales fp32 [heads, nb]).

    codes = Quantize(x / s) with the fp32 quotient x / s of the block's scale.
    """
    x = np.asarray(x, dtype=np.float32)
    s = block_scales(x, block_rows)
    per_row = np.repeat(s, block_rows, axis=1)[:, :x.shape[1]]
    y = (x / per_row[:, :, None]).astype(np.float32)   # fp32 division, per element
    return e4m3_encode(y), s


def dequantize_blocks(codes, scales, block_rows=BLOCK_ROWS) -> np.ndarray:
    """codes * s per block, in float64 (exact: both factors are short)."""
    vals = e4m3_decode(codes)
    per_row = np.repeat(np.asarray(scales, dtype=np.float64), block_rows, axis=1)
    return vals * per_row[:, :vals.shape[1], None]
