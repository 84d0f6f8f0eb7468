"""Seeded synthetic inputs for the attention forward pass.

This module is the one piece of code that both the CUDA path and the
fp64 oracle consume.  It holds no attention arithmetic: it only draws
reproducible normal variates and rounds them to bfloat16 bit patterns.

Generator
---------
* Uniforms come from SplitMix64 (Steele, Lea & Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014; the constants are the
  published ones) used in counter mode: output ``c`` of stream ``seed`` is
  ``mix64(seed * PHI + (c + 1) * PHI)`` with ``PHI = 0x9E3779B97F4A7C15``.
  A 64-bit output ``z`` becomes the uniform ``((z >> 11) + 1) * 2**-53``
  in (0, 1].
* Normals come from the Box-Muller transform: variate pair ``p`` uses
  uniforms ``2p`` and ``2p + 1``; element ``2p`` takes the cosine branch,
  element ``2p + 1`` the sine branch.
* Q, K and V are drawn in that order from ONE counter stream, element-major
  over ``[B, H, L, d]``: Q takes counters ``[0, n)``, K ``[n, 2n)``,
  V ``[2n, 3n)`` where ``n = B*H*L*d``.  The output gradient dO of the
  backward pass (standard deviation 1) takes ``[3n, 4n)``.
* Each variate is multiplied by its tensor's standard deviation, rounded to
  float32 (round-to-nearest-even) and then to bfloat16 (round-to-nearest-
  even on the float32 bit pattern).

Being counter based, any element can be regenerated on its own, so a test
can rebuild a few rows of a multi-gigabyte workload without drawing the
rest.
"""

from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os

import numpy as np

__all__ = [
    "AttentionWorkload",
    "WORKLOADS",
    "splitmix64_uniform",
    "normal_variates",
    "round_to_bf16_bits",
    "bf16_bits_to_float32",
    "make_qkv",
    "make_qkv_rows",
    "make_grad_out",
    "make_grad_out_rows",
    "make_custom_grad_out",
]

_PHI = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22  # elements per generation chunk (bounds host memory)


@dataclasses.dataclass(frozen=True)
class AttentionWorkload:
    """One synthetic attention forward problem: shapes, mask, scale, law."""

    name: str
    B: int
    H: int
    L: int
    d: int
    causal: bool
    scale: float
    seed: int
    q_std: float = 1.0
    k_std: float = 1.0
    v_std: float = 1.0

    @property
    def n_elem(self) -> int:
        return self.B * self.H * self.L * self.d

    @property
    def flops(self) -> float:
        """4*B*H*L^2*d, halved when causal (the metric's convention)."""
        f = 4.0 * self.B * self.H * self.L * self.L * self.d
        return f / 2.0 if self.causal else f

    @property
    def algorithmic_bytes(self) -> int:
        """Read Q, K, V once (bf16), write O (bf16) and LSE (fp32) once."""
        return 4 * self.n_elem * 2 + 4 * self.B * self.H * self.L


def _w(name, B, H, L, d, causal, scale, seed, qk_std=1.0):
    return AttentionWorkload(name, B, H, L, d, causal, scale, seed,
                             q_std=qk_std, k_std=qk_std, v_std=1.0)


#: The synthetic workloads.  Seed = 42 + index.  ``gate_d128_L8192`` is the
#: d=128 non-causal long-sequence point on which the tensor-core fraction is
#: judged (none of the others is d=128 and non-causal).
WORKLOADS = {
    w.name: w
    for w in (
        _w("single_head_L128_d64", 1, 1, 128, 64, False, 1.0 / math.sqrt(64), 42),
        _w("B4_H8_L1024_d64", 4, 8, 1024, 64, False, 1.0 / 8.0, 43),
        _w("B2_H16_L4096_d128_causal", 2, 16, 4096, 128, True, 1.0 / math.sqrt(128), 44),
        _w("B1_H32_L16384_d128_causal_qk3", 1, 32, 16384, 128, True,
           1.0 / math.sqrt(128), 45, qk_std=3.0),
        _w("B1_H16_L32768_d64", 1, 16, 32768, 64, False, 1.0 / 8.0, 46),
        _w("gate_B1_H32_L8192_d128", 1, 32, 8192, 128, False, 1.0 / math.sqrt(128), 47),
    )
}


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64_uniform(seed: int, counters: np.ndarray) -> np.ndarray:
    """Uniforms in (0, 1] for the given uint64 counters of stream ``seed``."""
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        base = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) * _PHI
        z = _mix64(base + (c + np.uint64(1)) * _PHI)
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def normal_variates(seed: int, start: int, count: int) -> np.ndarray:
    """Standard normals for element counters ``[start, start + count)``."""
    if count <= 0:
        return np.zeros(0, dtype=np.float64)
    first_pair = start // 2
    last_pair = (start + count - 1) // 2
    pairs = np.arange(first_pair, last_pair + 1, dtype=np.uint64)
    u1 = splitmix64_uniform(seed, pairs * np.uint64(2))
    u2 = splitmix64_uniform(seed, pairs * np.uint64(2) + np.uint64(1))
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * np.pi * u2
    out = np.empty(2 * pairs.size, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    off = start - 2 * first_pair
    return out[off:off + count]


def normal_at(seed: int, counters: np.ndarray) -> np.ndarray:
    """Standard normals at arbitrary (not necessarily contiguous) counters."""
    c = np.asarray(counters, dtype=np.uint64)
    pair = c // np.uint64(2)
    u1 = splitmix64_uniform(seed, pair * np.uint64(2))
    u2 = splitmix64_uniform(seed, pair * np.uint64(2) + np.uint64(1))
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * np.pi * u2
    return np.where((c & np.uint64(1)) == 0, r * np.cos(t), r * np.sin(t))


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64/float32 -> bfloat16 bit patterns (uint16), RNE via float32."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    out = rounded.astype(np.uint16)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_float32(b: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _fill(seed: int, start: int, n: int, std: float) -> np.ndarray:
    """Counters ``[start, start + n)`` as bf16 bits.  Chunks are independent
    (counter mode), so they are drawn on a thread pool: numpy releases the
    interpreter lock inside its array operations, and every chunk's values
    depend only on its counters, so the result is the same for any thread
    count."""
    out = np.empty(n, dtype=np.uint16)

    def chunk(lo):
        hi = min(n, lo + _CHUNK)
        out[lo:hi] = round_to_bf16_bits(std * normal_variates(seed, start + lo, hi - lo))

    starts = range(0, n, _CHUNK)
    workers = min(len(starts), os.cpu_count() or 1)
    if workers <= 1:
        for lo in starts:
            chunk(lo)
    else:
        with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as pool:
            list(pool.map(chunk, starts))
    return out


def make_qkv(w: AttentionWorkload):
    """Q, K, V as bf16 bit patterns, each a uint16 array of shape [B,H,L,d]."""
    n = w.n_elem
    shape = (w.B, w.H, w.L, w.d)
    q = _fill(w.seed, 0, n, w.q_std).reshape(shape)
    k = _fill(w.seed, n, n, w.k_std).reshape(shape)
    v = _fill(w.seed, 2 * n, n, w.v_std).reshape(shape)
    return q, k, v


def make_qkv_rows(w: AttentionWorkload, bh: int, rows: np.ndarray):
    """Rebuild rows ``rows`` of head ``bh`` (= b*H + h) of Q, K and V.

    Returns three uint16 arrays of shape [len(rows), d], bit-identical to
    the corresponding rows of :func:`make_qkv`.
    """
    n = w.n_elem
    rows = np.asarray(rows, dtype=np.int64)
    base = (bh * w.L + rows)[:, None] * w.d + np.arange(w.d, dtype=np.int64)[None, :]
    base = base.astype(np.uint64)
    out = []
    for t, std in enumerate((w.q_std, w.k_std, w.v_std)):
        z = normal_at(w.seed, base + np.uint64(t * n))
        out.append(round_to_bf16_bits(std * z).reshape(rows.size, w.d))
    return tuple(out)


def make_grad_out(w: AttentionWorkload):
    """The output gradient dO (bf16 bits [B,H,L,d], standard normal)."""
    n = w.n_elem
    return _fill(w.seed, 3 * n, n, 1.0).reshape(w.B, w.H, w.L, w.d)


def make_grad_out_rows(w: AttentionWorkload, bh: int, rows: np.ndarray):
    """Rows ``rows`` of head ``bh`` of :func:`make_grad_out` ([len(rows), d])."""
    n = w.n_elem
    rows = np.asarray(rows, dtype=np.int64)
    base = (bh * w.L + rows)[:, None] * w.d + np.arange(w.d, dtype=np.int64)[None, :]
    z = normal_at(w.seed, base.astype(np.uint64) + np.uint64(3 * n))
    return round_to_bf16_bits(z).reshape(rows.size, w.d)


def make_custom_grad_out(B, H, L, d, seed):
    """dO for an ad-hoc shape, from the same stream as :func:`make_custom`."""
    return make_grad_out(AttentionWorkload("custom", B, H, L, d, False, 1.0, seed))


def make_custom(B, H, L, d, seed, q_std=1.0, k_std=1.0, v_std=1.0):
    """Q, K, V for an ad-hoc shape (tests sweeping ragged sizes)."""
    w = AttentionWorkload("custom", B, H, L, d, False, 1.0, seed, q_std, k_std, v_std)
    return make_qkv(w)
