"""GPU parity of the split-KV forward (split pass + merge) against the oracle.

Every call goes through the C ABI (``fa_fwd_splitkv`` via the binding).
Split-KV computes the same exact attention as ``fa_fwd``; the split count
only changes the order of the sums.
"""

from __future__ import annotations

import math

import numpy as np
import pytest

import exact_tiled_attention_09_gb300 as fa
from fa_inputs import bf16_bits_to_float32, make_custom
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
    assert fa.fa_device_status(None, clear=True) == fa.FA_OK, "a kernel wait timed out"


def _f64(bits):
    return bf16_bits_to_float32(bits).astype(np.float64)


def _split(dev, qb, kb, vb, scale, causal, n_splits, workspace=None):
    import torch
    q, k, v = (to_device(x, dev) for x in (qb, kb, vb))
    o, lse = fa.forward_splitkv(q, k, v, n_splits, scale=scale, causal=causal,
                                workspace=workspace)
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("n_splits", [1, 2, 3, 7, 64])
@pytest.mark.parametrize("L", [129, 1000, 1024])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_parity(dev, n_splits, L, d, causal):
    qb, kb, vb = make_custom(1, 2, L, d, seed=3000 + L + d + n_splits + int(causal))
    scale = 1.0 / math.sqrt(d)
    o, lse = _split(dev, qb, kb, vb, scale, causal, n_splits)
    o_ref, lse_ref, a_ref = oracle_forward(_f64(qb), _f64(kb), _f64(vb), scale, causal)
    check_parity(from_device(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                 f"split={n_splits} L={L} d={d} causal={causal}", absv_ref=a_ref)


@pytest.mark.parametrize("L", [1, 2, 127])
def test_splitkv_short_sequences(dev, L):
    # more splits requested than key blocks: the pass uses one split
    qb, kb, vb = make_custom(2, 3, L, 64, seed=77 + L)
    o, lse = _split(dev, qb, kb, vb, 0.125, True, 8)
    o_ref, lse_ref, a_ref = oracle_forward(_f64(qb), _f64(kb), _f64(vb), 0.125, True)
    check_parity(from_device(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                 f"short L={L}", absv_ref=a_ref)


@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_long_sequence_sampled(dev, causal):
    import torch
    B, H, L, d = 1, 4, 8192, 128
    qb, kb, vb = make_custom(B, H, L, d, seed=4242 + int(causal), q_std=2.0, k_std=2.0)
    o, lse = _split(dev, qb, kb, vb, 1.0 / math.sqrt(d), causal, 6)
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    rows = np.array([0, 1, 127, 128, 255, 256, 4095, 4096, 8190, 8191])
    for h in (0, 3):
        qh, kh, vh = (_f64(x[0, h]) for x in (qb, kb, vb))
        o_ref, lse_ref, a_ref = oracle_forward(qh, kh, vh, 1.0 / math.sqrt(d), causal, rows=rows)
        check_parity(from_device(o[0, h, rows]), lse[0, h, rows].cpu().numpy().astype(np.float64),
                     o_ref, lse_ref, f"L=8192 head {h} causal={causal}", absv_ref=a_ref)


def test_splitkv_matches_single_pass(dev):
    import torch
    qb, kb, vb = make_custom(2, 4, 2000, 64, seed=9)
    q, k, v = (to_device(x, dev) for x in (qb, kb, vb))
    o1, l1 = fa.forward(q, k, v, scale=0.125)
    o2, l2 = fa.forward_splitkv(q, k, v, 5, scale=0.125)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 1e-4


def test_splitkv_workspace_reuse(dev):
    import torch
    L, d, S = 700, 128, 4
    ws = torch.empty(fa.fa_splitkv_workspace_bytes(1, 2, L, d, S), dtype=torch.uint8, device=dev)
    for seed in (1, 2):
        qb, kb, vb = make_custom(1, 2, L, d, seed=seed)
        o, lse = _split(dev, qb, kb, vb, 0.1, bool(seed % 2), S, workspace=ws)
        o_ref, lse_ref, a_ref = oracle_forward(_f64(qb), _f64(kb), _f64(vb), 0.1, bool(seed % 2))
        check_parity(from_device(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                     f"reuse seed {seed}", absv_ref=a_ref)


def test_splitkv_back_to_back_calls_share_one_workspace(dev):
    # Two split-KV calls on one stream without a host sync, one workspace:
    # the merge is a programmatic dependant of its split pass; the second
    # call's split pass must not overwrite partials the first merge still
    # reads.
    import torch
    L, d, S = 900, 64, 5
    ws = torch.empty(fa.fa_splitkv_workspace_bytes(2, 2, L, d, S), dtype=torch.uint8,
                     device=dev)
    cases = [make_custom(2, 2, L, d, seed=seed) for seed in (31, 32)]
    outs = []
    for qb, kb, vb in cases:
        q, k, v = (to_device(x, dev) for x in (qb, kb, vb))
        outs.append(fa.forward_splitkv(q, k, v, S, scale=0.125, causal=False, workspace=ws))
    torch.cuda.synchronize()
    for (qb, kb, vb), (o, lse) in zip(cases, outs):
        o_ref, lse_ref, a_ref = oracle_forward(_f64(qb), _f64(kb), _f64(vb), 0.125, False)
        check_parity(from_device(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                     "back to back", absv_ref=a_ref)


def test_splitkv_recommended_split_count(dev):
    # n_splits=None takes the library's recommendation for the current GPU
    import torch
    L, d = 3000, 128
    qb, kb, vb = make_custom(1, 1, L, d, seed=41)
    S = fa.fa_splitkv_splits(1, 1, L, d, True)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    assert S == fa.fa_splitkv_splits(1, 1, L, d, True, sms) and S > 1
    q, k, v = (to_device(x, dev) for x in (qb, kb, vb))
    o, lse = fa.forward_splitkv(q, k, v, scale=0.09, causal=True)
    torch.cuda.synchronize()
    o_ref, lse_ref, a_ref = oracle_forward(_f64(qb), _f64(kb), _f64(vb), 0.09, True)
    check_parity(from_device(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                 "recommended splits", absv_ref=a_ref)
