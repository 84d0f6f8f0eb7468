"""GPU parity of the FP8 forward and its block quantisation.

The quantisation kernel must reproduce the oracle's E4M3 codes and block
scales bit for bit (integer work, decisions taken in fp32 on both sides).
The FP8 forward must match exact attention of the de-quantised Q and K with
V (the oracle's fp64 forward on codes x block scale) within the forward's
tolerances.  Every call goes through the C ABI.
"""

from __future__ import annotations

import math

import numpy as np
import pytest

import exact_tiled_attention_09_gb300 as fa
import oracle
from oracle import fp8 as ofp8
from fa_inputs import WORKLOADS, bf16_bits_to_float32, make_custom, make_qkv, round_to_bf16_bits
from tests.gpu_util import check_parity, oracle_forward, from_device, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.library()
    fa.fa_device_status(None, clear=True)
    yield torch.device("cuda:0")
    assert fa.fa_device_status(None, clear=True) == fa.FA_OK


def _f32(bits):
    return bf16_bits_to_float32(bits)


def _quant_gpu(dev, bits):
    import torch
    codes, scales = fa.quantize_fp8(to_device(bits, dev))
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("L", [1, 127, 128, 300, 1000])
@pytest.mark.parametrize("d", [64, 128])
def test_quantisation_is_bit_exact(dev, L, d):
    qb, kb, _ = make_custom(2, 3, L, d, 4000 + L + d, q_std=1.0, k_std=7.0)
    for bits in (qb, kb):
        codes, scales = _quant_gpu(dev, bits)
        x = _f32(bits).reshape(6, L, d)
        ref_codes, ref_scales = ofp8.quantize_blocks(x)
        assert np.array_equal(scales.reshape(ref_scales.shape).view(np.uint32),
                              ref_scales.view(np.uint32))
        got = codes.reshape(ref_codes.shape)
        bad = got != ref_codes
        assert not bad.any(), (f"{int(bad.sum())} codes differ, e.g. x={x[bad][:4]} "
                               f"got={got[bad][:4]} want={ref_codes[bad][:4]}")


def test_quantisation_edge_values(dev):
    # zeros (scale 1), a zero block next to a live one, wide dynamic range
    # (subnormal codes), exact powers of two, negative values and -0
    L, d = 256, 64
    x = np.zeros((1, 1, L, d), np.float32)
    rng = np.random.default_rng(3)
    x[0, 0, 128:] = rng.standard_normal((128, d)) * np.exp2(rng.integers(-20, 8, (128, d)))
    x[0, 0, 130, :8] = [448.0, -448.0, 2.0 ** -30, -0.0, 1.0, -1.0, 0.5, 2.0 ** 7]
    bits = round_to_bf16_bits(x)
    codes, scales = _quant_gpu(dev, bits)
    ref_codes, ref_scales = ofp8.quantize_blocks(_f32(bits).reshape(1, L, d))
    assert np.array_equal(scales.reshape(1, 2).view(np.uint32), ref_scales.view(np.uint32))
    assert np.array_equal(codes.reshape(1, L, d), ref_codes)


def _host_quantised(bits, BH, L, d):
    """The oracle's E4M3 codes and block scales of a bf16 input, quantised on
    the host from the input itself (never from the GPU's codes)."""
    return ofp8.quantize_blocks(_f32(bits).reshape(BH, L, d))


def _assert_same_codes(dev_codes, dev_scales, ref_codes, ref_scales, label):
    got_c = dev_codes.cpu().numpy().reshape(ref_codes.shape)
    got_s = dev_scales.cpu().numpy().reshape(ref_scales.shape).astype(np.float32)
    assert np.array_equal(got_s.view(np.uint32), ref_scales.astype(np.float32).view(np.uint32)), \
        f"{label}: block scales differ from the oracle's"
    bad = got_c != ref_codes
    assert not bad.any(), f"{label}: {int(bad.sum())} E4M3 codes differ from the oracle's"


def _fp8_case(dev, qb, kb, vb, scale, causal, label, config=None):
    import torch
    B, H, L, d = qb.shape
    BH = B * H
    q, k, v = (to_device(x, dev) for x in (qb, kb, vb))
    q8, qs = fa.quantize_fp8(q)
    k8, ks = fa.quantize_fp8(k)
    o, lse = fa.forward_fp8(q8, k8, v, qs, ks, scale=scale, causal=causal)
    torch.cuda.synchronize()
    # expected result: exact attention of the oracle's own quantisation of
    # the host inputs; the GPU's codes must equal those bit for bit
    qc, qsc = _host_quantised(qb, BH, L, d)
    kc, ksc = _host_quantised(kb, BH, L, d)
    _assert_same_codes(q8, qs, qc, qsc, label + " Q")
    _assert_same_codes(k8, ks, kc, ksc, label + " K")
    qd = ofp8.dequantize_blocks(qc, qsc)
    kd = ofp8.dequantize_blocks(kc, ksc)
    vd = _f32(vb).astype(np.float64).reshape(BH, L, d)
    o_ref, lse_ref, a_ref = oracle_forward(qd, kd, vd, scale, causal)
    return check_parity(from_device(o).reshape(BH, L, d),
                        lse.cpu().numpy().astype(np.float64).reshape(BH, L),
                        o_ref, lse_ref, label, config, absv_ref=a_ref)


@pytest.mark.parametrize("L", [1, 17, 128, 129, 300, 1000])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_ragged(dev, L, d, causal):
    qb, kb, vb = make_custom(1, 2, L, d, 4100 + L + d + int(causal))
    _fp8_case(dev, qb, kb, vb, 1.0 / math.sqrt(d), causal, f"fp8 L={L} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_forward_batch_heads_and_scales(dev, d):
    qb, kb, vb = make_custom(3, 2, 400, d, 4200 + d, q_std=3.0, k_std=3.0)
    for scale in (1.0 / math.sqrt(d), -0.2, 0.0):
        for causal in (False, True):
            _fp8_case(dev, qb, kb, vb, scale, causal, f"fp8 d={d} scale={scale} causal={causal}")


def test_fp8_forward_benchmark_workload(dev):
    w = WORKLOADS["B4_H8_L1024_d64"]
    qb, kb, vb = make_qkv(w)
    _fp8_case(dev, qb, kb, vb, w.scale, w.causal, "fp8 " + w.name, config="fp8 " + w.name)


@pytest.mark.parametrize("name", ["gate_B1_H32_L8192_d128", "B1_H32_L16384_d128_causal_qk3",
                                  "B1_H16_L32768_d64"])
def test_fp8_forward_full_size_sampled(dev, name):
    import torch
    w = WORKLOADS[name]
    qb, kb, vb = make_qkv(w)
    BH = w.B * w.H
    q, k, v = (to_device(x, dev) for x in (qb, kb, vb))
    q8, qs = fa.quantize_fp8(q)
    k8, ks = fa.quantize_fp8(k)
    o, lse = fa.forward_fp8(q8, k8, v, qs, ks, scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    rng = np.random.default_rng(w.seed)
    rows = sorted({0, 1, 127, 128, w.L // 2, w.L - 1} | set(int(x) for x in rng.integers(0, w.L, 8)))
    qf, kf, vf = (x.reshape(BH, w.L, w.d) for x in (qb, kb, vb))
    for h in (0, BH - 1):
        # the oracle quantises this head's Q and K from the host inputs
        qc, qsc = _host_quantised(qf[h], 1, w.L, w.d)
        kc, ksc = _host_quantised(kf[h], 1, w.L, w.d)
        _assert_same_codes(q8.view(BH, w.L, w.d)[h], qs.view(BH, -1)[h], qc, qsc,
                           f"fp8 {name} head {h} Q")
        _assert_same_codes(k8.view(BH, w.L, w.d)[h], ks.view(BH, -1)[h], kc, ksc,
                           f"fp8 {name} head {h} K")
        qd = ofp8.dequantize_blocks(qc, qsc)[0]
        kd = ofp8.dequantize_blocks(kc, ksc)[0]
        o_ref, lse_ref, a_ref = oracle_forward(qd, kd, _f32(vf[h]).astype(np.float64), w.scale,
                                          w.causal, rows=rows)
        check_parity(from_device(o.view(BH, w.L, w.d)[h, rows]),
                     lse.view(BH, w.L)[h, rows].cpu().numpy().astype(np.float64), o_ref, lse_ref,
                     f"fp8 {name} head {h}", config="fp8 " + name, absv_ref=a_ref)
