"""Pins for the FP8 (E4M3) block quantisation of the oracle.

Pinned to the format's definition (1-4-3 bits, bias 7, subnormals m * 2^-9,
max 448, no infinities) by brute force over the 254 finite values, and to
the quantisation formula of "FlashAttention 深度解析", third part, section
2.3: s = max|block| / FP8_MAX and S = (Q_FP8 K_FP8^T) s_q s_k.  Planted
mistakes in a copy of the encoder must fail the same checks.
"""

from __future__ import annotations

import numpy as np
import pytest

from oracle import fp8


def _table():
    """All finite E4M3 values from the bit-field definition, by code."""
    vals = {}
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 0x7
        if e == 0xF and m == 0x7:
            continue
        vals[c] = s * (m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return vals


def _brute_encode(x):
    """Nearest finite value (ties: even mantissa bit), saturating; +0 for 0."""
    t = _table()
    out = []
    for v in np.asarray(x, dtype=np.float64).ravel():
        v = min(max(v, -448.0), 448.0)
        best = None
        for c, w in t.items():
            if (c & 0x80) != (0x80 if np.signbit(v) else 0):
                continue
            dist = abs(w - v)
            if best is None or dist < best[0] - 1e-300 or (dist == best[0] and (c & 1) == 0):
                best = (dist, c)
        out.append(best[1])
    return np.array(out, dtype=np.uint8)


def encoder_pins_pass(enc) -> bool:
    t = _table()
    codes = np.array(sorted(t), dtype=np.uint8)
    vals = np.array([t[c] for c in codes])
    if not np.array_equal(enc(vals), codes):
        return False
    # every midpoint between neighbours, and random values
    pos = np.array(sorted(v for v in vals if v >= 0))
    mids = (pos[:-1] + pos[1:]) / 2
    rng = np.random.default_rng(5)
    samples = np.concatenate([mids, -mids, rng.uniform(-600, 600, 400),
                              rng.uniform(-0.05, 0.05, 400), [0.0, 1e6, -1e6, 2.0 ** -11]])
    return bool(np.array_equal(enc(samples), _brute_encode(samples)))


def test_format_constants():
    d = fp8.e4m3_decode(np.array([0x38, 0x7E, 0x01, 0x07, 0x08, 0x78, 0xB8, 0x00], np.uint8))
    assert list(d) == [1.0, 448.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 256.0, -1.0, 0.0]
    assert np.isnan(fp8.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    mags = fp8.e4m3_decode(np.arange(0, 127, dtype=np.uint8))
    assert np.all(np.diff(mags) > 0)


def test_encoder_matches_brute_force():
    assert encoder_pins_pass(fp8.e4m3_encode)


def test_saturation_and_nan():
    c = fp8.e4m3_encode(np.array([448.0, 464.0, 1e30, -1e30, np.nan]))
    assert list(c[:4]) == [0x7E, 0x7E, 0x7E, 0xFE] and c[4] == 0x7F


@pytest.mark.parametrize("mutation", ["half_away", "bias8", "truncate"])
def test_encoder_mutants_fail(mutation):
    def bad(x):
        x = np.asarray(x, dtype=np.float64)
        if mutation == "half_away":
            # ties away from zero instead of to even
            return fp8.e4m3_encode(x + np.sign(x) * np.abs(x) * 1e-12)
        if mutation == "bias8":
            return fp8.e4m3_encode(x * 2.0)
        return fp8.e4m3_encode(np.sign(x) * np.abs(x) * (1 - 2.0 ** -5))
    assert not encoder_pins_pass(bad)


def test_block_scale_maps_amax_to_fp8_max():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((3, 300, 64)) * rng.uniform(0.01, 50, (3, 300, 1))).astype(np.float32)
    codes, s = fp8.quantize_blocks(x)
    assert s.shape == (3, 3) and s.dtype == np.float32
    for h in range(3):
        for b in range(3):
            blk = x[h, b * 128:(b + 1) * 128]
            amax = np.abs(blk).max()
            assert s[h, b] == np.float32(amax) / np.float32(448.0)
            cb = codes[h, b * 128:(b + 1) * 128]
            i = np.unravel_index(np.abs(blk).argmax(), blk.shape)
            assert abs(fp8.e4m3_decode(cb[i])) == 448.0


def test_dequantisation_error_is_half_a_quantum():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((2, 256, 128)).astype(np.float32) * 3
    codes, s = fp8.quantize_blocks(x)
    deq = fp8.dequantize_blocks(codes, s)
    sr = np.repeat(s.astype(np.float64), 128, axis=1)[:, :, None]
    y = np.abs(x.astype(np.float64)) / sr          # magnitude in code units
    quantum = np.where(y >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(y, 2.0 ** -6))) - 3),
                       2.0 ** -9)
    # half a quantum in code units, plus the fp32 rounding of x / s
    assert np.all(np.abs(deq - x) <= (quantum / 2) * sr * (1 + 2.0 ** -20) + 1e-30)


def test_zero_block_and_ragged_tail():
    x = np.zeros((1, 130, 64), np.float32)
    x[0, 128:, :] = 1.5
    codes, s = fp8.quantize_blocks(x)
    assert s[0, 0] == 1.0 and not codes[0, :128].any()
    assert s[0, 1] == np.float32(1.5) / np.float32(448.0)
    assert (fp8.e4m3_decode(codes[0, 128:]) == 448.0).all()


def test_dequantised_scores_equal_the_pages_formula():
    # S = (Q_FP8 K_FP8^T) * s_q * s_k, evaluated block by block, equals the
    # product of the de-quantised inputs (exact in fp64 at these sizes)
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 256, 64)).astype(np.float32)
    k = (rng.standard_normal((1, 256, 64)) * 4).astype(np.float32)
    qc, sq = fp8.quantize_blocks(q)
    kc, sk = fp8.quantize_blocks(k)
    s_blocks = np.zeros((256, 256))
    for i in range(2):
        for j in range(2):
            qa = fp8.e4m3_decode(qc[0, i * 128:(i + 1) * 128])
            ka = fp8.e4m3_decode(kc[0, j * 128:(j + 1) * 128])
            s_blocks[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128] = \
                (qa @ ka.T) * float(sq[0, i]) * float(sk[0, j])
    s_deq = fp8.dequantize_blocks(qc, sq)[0] @ fp8.dequantize_blocks(kc, sk)[0].T
    assert np.allclose(s_blocks, s_deq, rtol=1e-14, atol=1e-12)
