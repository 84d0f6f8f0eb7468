"""GPU parity: the sm_103a kernel against the fp64 oracle, element by element.

Every call goes through the C ABI (``fa_fwd`` via the ctypes binding).
Small problems are compared in full; the full-size workloads are run in the
same launch configuration the benchmark uses and compared on sampled rows
that the oracle computes one by one (first and last rows, rows around tile
boundaries, random rows, several heads).
"""

from __future__ import annotations

import math

import numpy as np
import pytest

import exact_tiled_attention_09_gb300 as fa
import oracle
from fa_inputs import WORKLOADS, bf16_bits_to_float32, make_custom, make_qkv
from tests.gpu_util import check_parity, oracle_forward, from_device, o_tolerance, to_device

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


def _run(dev, qb, kb, vb, scale, causal):
    import torch
    q, k, v = (to_device(x, dev) for x in (qb, kb, vb))
    o, lse = fa.forward(q, k, v, scale=scale, causal=causal)
    torch.cuda.synchronize()
    return o, lse


def _full_parity(dev, qb, kb, vb, scale, causal, label, config=None):
    o, lse = _run(dev, qb, kb, vb, scale, causal)
    o_ref, lse_ref, a_ref = oracle_forward(_f64(qb), _f64(kb), _f64(vb), scale, causal)
    return check_parity(from_device(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                        label, config, absv_ref=a_ref)


# ------------------------------------------------------------------ workloads
@pytest.mark.parametrize("name", ["single_head_L128_d64", "B4_H8_L1024_d64"])
def test_workload_full(dev, name):
    w = WORKLOADS[name]
    qb, kb, vb = make_qkv(w)
    _full_parity(dev, qb, kb, vb, w.scale, w.causal, name, config=name)


def _sample_rows(L, rng, n_random=12):
    rows = {0, 1, 2, 127, 128, 129, L // 2, L - 129, L - 128, L - 2, L - 1}
    rows |= set(int(x) for x in rng.integers(0, L, n_random))
    return sorted(r for r in rows if 0 <= r < L)


@pytest.mark.parametrize("name", ["B2_H16_L4096_d128_causal", "gate_B1_H32_L8192_d128",
                                  "B1_H16_L32768_d64", "B1_H32_L16384_d128_causal_qk3"])
def test_workload_full_size_sampled(dev, name):
    import torch
    w = WORKLOADS[name]
    qb, kb, vb = make_qkv(w)
    o, lse = _run(dev, qb, kb, vb, w.scale, w.causal)
    o_h = o.view(w.B * w.H, w.L, w.d)
    lse_h = lse.view(w.B * w.H, w.L)
    assert bool(torch.isfinite(o_h).all()) and bool(torch.isfinite(lse_h).all())
    rng = np.random.default_rng(w.seed)
    BH = w.B * w.H
    heads = sorted({0, BH - 1} | set(int(x) for x in rng.integers(0, BH, 3)))
    qf, kf, vf = (x.reshape(BH, w.L, w.d) for x in (qb, kb, vb))
    for h in heads:
        rows = _sample_rows(w.L, rng)
        o_ref, lse_ref, a_ref = oracle_forward(_f64(qf[h]), _f64(kf[h]), _f64(vf[h]), w.scale,
                                          w.causal, rows=rows)
        o_gpu = from_device(o_h[h, rows])
        lse_gpu = lse_h[h, rows].cpu().numpy().astype(np.float64)
        check_parity(o_gpu, lse_gpu, o_ref, lse_ref, f"{name} head {h}", config=name, absv_ref=a_ref)


# ------------------------------------------------------------------ shapes
@pytest.mark.parametrize("L", [1, 2, 15, 16, 17, 127, 128, 129, 255, 257, 1000])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(dev, L, d, causal):
    qb, kb, vb = make_custom(1, 2, L, d, seed=1000 + L + d + int(causal))
    _full_parity(dev, qb, kb, vb, 1.0 / math.sqrt(d), causal, f"L={L} d={d} causal={causal}")


@pytest.mark.parametrize("B,H", [(1, 1), (3, 5), (2, 1), (1, 7)])
@pytest.mark.parametrize("d", [64, 128])
def test_batch_head_edges(dev, B, H, d):
    qb, kb, vb = make_custom(B, H, 200, d, seed=77 + B * 10 + H)
    _full_parity(dev, qb, kb, vb, 1.0 / math.sqrt(d), False, f"B={B} H={H} d={d}")
    _full_parity(dev, qb, kb, vb, 1.0 / math.sqrt(d), True, f"B={B} H={H} d={d} causal")


@pytest.mark.parametrize("scale", [0.0, 2.0, -0.3, 1e-3])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_scales(dev, scale, d, causal):
    qb, kb, vb = make_custom(1, 2, 300, d, seed=500 + d)
    _full_parity(dev, qb, kb, vb, scale, causal, f"scale={scale} d={d} causal={causal}")


def test_large_logits_rescale_path(dev):
    # Q, K ~ N(0, 3^2) with d=128: scores of tens, the running max keeps growing
    qb, kb, vb = make_custom(1, 4, 1500, 128, seed=901, q_std=3.0, k_std=3.0)
    for causal in (False, True):
        _full_parity(dev, qb, kb, vb, 1.0 / math.sqrt(128), causal, f"qk3 causal={causal}")


def test_increasing_max_forces_every_rescale(dev):
    # key j has score growing with j: every K/V block raises the row max by
    # much more than the rescale threshold.
    L, d = 640, 64
    q = np.zeros((1, 1, L, d), np.float32); q[..., 0] = 1.0
    k = np.zeros((1, 1, L, d), np.float32)
    k[0, 0, :, 0] = np.linspace(0, 60, L)
    v = np.random.default_rng(3).standard_normal((1, 1, L, d)).astype(np.float32)
    from fa_inputs import round_to_bf16_bits
    qb, kb, vb = (round_to_bf16_bits(x) for x in (q, k, v))
    for causal in (False, True):
        _full_parity(dev, qb, kb, vb, 1.0, causal, f"growing max causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_max_growth_around_the_rescale_threshold(dev, d):
    # Row r's score for key j is a_r * c * j with a_r from 0.2 to 1.0: per
    # block of 128 keys the max grows by up to ~5.8 powers of two, so rows
    # keep a stale reference (P~ above 1) for a block or two and then
    # rescale, each at its own block; a warp mixes rows that need the
    # rescale with rows that do not.
    L = 1000
    per_block = 5.8 / math.log2(math.e)           # score growth per block
    q = np.zeros((1, 2, L, d), np.float32)
    q[..., 0] = np.linspace(0.2, 1.0, L)
    k = np.zeros((1, 2, L, d), np.float32)
    k[..., 0] = np.arange(L) * (per_block / 128.0)
    rng = np.random.default_rng(17)
    q[..., 1:] = 0.05 * rng.standard_normal((1, 2, L, d - 1))
    k[..., 1:] = 0.05 * rng.standard_normal((1, 2, L, d - 1))
    v = rng.standard_normal((1, 2, L, d)).astype(np.float32)
    from fa_inputs import round_to_bf16_bits
    qb, kb, vb = (round_to_bf16_bits(x) for x in (q, k, v))
    for causal in (False, True):
        _full_parity(dev, qb, kb, vb, 1.0, causal, f"threshold growth d={d} causal={causal}")


# ------------------------------------------------------------------ invariants
def test_causal_first_row_is_v0_exactly(dev):
    qb, kb, vb = make_custom(2, 3, 300, 128, seed=31)
    o, lse = _run(dev, qb, kb, vb, 0.1, True)
    o0 = o[:, :, 0].cpu().reshape(-1)
    v0 = to_device(vb, "cpu")[:, :, 0].reshape(-1)
    assert bool((o0 == v0).all())
    s00 = 0.1 * np.einsum("bhd,bhd->bh", _f64(qb)[:, :, 0], _f64(kb)[:, :, 0])
    assert np.abs(lse[:, :, 0].cpu().numpy() - s00).max() <= 1e-4


def test_identical_value_rows(dev):
    L, d = 400, 64
    qb, kb, _ = make_custom(1, 2, L, d, seed=41)
    row = np.linspace(-3, 3, d).astype(np.float32)
    from fa_inputs import round_to_bf16_bits
    vb = round_to_bf16_bits(np.broadcast_to(row, (1, 2, L, d)).copy())
    o, _ = _run(dev, qb, kb, vb, 0.125, False)
    ref = bf16_bits_to_float32(vb).astype(np.float64)
    err = np.abs(from_device(o) - ref)
    # every row of V is the same, so A = sum_j p_ij |v_jc| = |v_c| exactly
    assert (err <= o_tolerance(ref, np.abs(ref))).all(), f"max err {err.max():.3e}"


def test_deterministic_bitwise(dev):
    w = WORKLOADS["B4_H8_L1024_d64"]
    qb, kb, vb = make_qkv(w)
    o1, l1 = _run(dev, qb, kb, vb, w.scale, False)
    o2, l2 = _run(dev, qb, kb, vb, w.scale, False)
    import torch
    assert bool((o1.view(torch.int16) == o2.view(torch.int16)).all())
    assert bool((l1 == l2).all())


def test_outputs_fully_overwritten(dev):
    import torch
    qb, kb, vb = make_custom(1, 2, 333, 64, seed=55)
    q, k, v = (to_device(x, dev) for x in (qb, kb, vb))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((1, 2, 333), float("nan"), device=dev)
    fa.forward(q, k, v, scale=0.125, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L", [129, 300])
def test_no_write_past_the_outputs(dev, d, causal, L):
    # O leaves through a tile-sized store whose rows past L are clipped by
    # the tensor map: nothing may land past the caller's buffer
    import torch
    qb, kb, vb = make_custom(1, 1, L, d, seed=66 + L + d)
    q, k, v = (to_device(x, dev) for x in (qb, kb, vb))
    o_big = torch.full((L + 256, d), 7.0, dtype=torch.bfloat16, device=dev)
    lse_big = torch.full((L + 256,), 7.0, device=dev)
    fa.forward(q, k, v, scale=0.125, causal=causal, out=o_big[:L].view(1, 1, L, d),
               lse=lse_big[:L].view(1, 1, L))
    torch.cuda.synchronize()
    assert bool((o_big[L:] == 7.0).all()) and bool((lse_big[L:] == 7.0).all())
    assert bool(torch.isfinite(o_big[:L]).all())


def test_status_after_runs_is_ok(dev):
    assert fa.fa_device_status(None, clear=False) == fa.FA_OK


# ------------------------------------------------------------------ scheduling
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_many_heads_in_several_scheduling_groups(dev, d, causal):
    # 960 heads of L = 256: heads are scheduled in groups whose K and V fit
    # in ~32 MB of L2 (512 heads a group at d = 64, 256 at d = 128), so
    # this covers several groups, a ragged last group and, causal, the
    # longest-first order across the heads of a group; every head in full
    B, H, L = 15, 64, 256
    qb, kb, vb = make_custom(B, H, L, d, seed=1300 + d + int(causal))
    _full_parity(dev, qb, kb, vb, 1.0 / math.sqrt(d), causal,
                 f"B={B} H={H} L={L} d={d} causal={causal}")


@pytest.mark.parametrize("L,d,causal", [(65536, 64, False), (40000, 128, True)])
def test_one_very_long_head_sampled(dev, L, d, causal):
    # one head, far longer than the workloads: 256-512 key blocks per CTA
    import torch
    qb, kb, vb = make_custom(1, 1, L, d, seed=1400 + d)
    o, lse = _run(dev, qb, kb, vb, 1.0 / math.sqrt(d), causal)
    rng = np.random.default_rng(L)
    rows = _sample_rows(L, rng, n_random=10)
    f = lambda x: _f64(x.reshape(L, d))
    o_ref, lse_ref, a_ref = oracle_forward(f(qb), f(kb), f(vb), 1.0 / math.sqrt(d), causal,
                                           rows=rows)
    check_parity(from_device(o.view(L, d)[rows]), lse.view(L)[rows].cpu().numpy().astype(np.float64),
                 o_ref, lse_ref, f"L={L} d={d} causal={causal}", absv_ref=a_ref)


def test_concurrent_streams(dev):
    # The kernels keep no state between calls (the status word aside): two
    # forwards and two backwards in flight at once on two streams, each on
    # its own inputs and workspace, match the oracle.
    import torch
    from fa_inputs import make_custom_grad_out
    L, d = 700, 64
    cases = [make_custom(2, 3, L, d, seed=1600 + i) for i in range(2)]
    dos = [make_custom_grad_out(2, 3, L, d, 1600 + i) for i in range(2)]
    streams = [torch.cuda.Stream(device=dev) for _ in range(2)]
    outs = []
    for (qb, kb, vb), dob, st in zip(cases, dos, streams):
        with torch.cuda.stream(st):
            q, k, v, do = (to_device(x, dev) for x in (qb, kb, vb, dob))
            o, lse = fa.forward(q, k, v, scale=0.125, causal=True, stream=st)
            grads = fa.backward(q, k, v, o, lse, do, scale=0.125, causal=True, stream=st)
            outs.append((o, lse, grads))
    torch.cuda.synchronize()
    from tests.gpu_util import check_grads_per_head
    for (qb, kb, vb), dob, (o, lse, grads) in zip(cases, dos, outs):
        o_ref, lse_ref, a_ref = oracle_forward(_f64(qb), _f64(kb), _f64(vb), 0.125, True)
        check_parity(from_device(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                     "concurrent streams", absv_ref=a_ref)
        ref = oracle.attention_bwd(_f64(qb), _f64(kb), _f64(vb), _f64(dob), 0.125, True)
        check_grads_per_head([from_device(t) for t in grads], ref, "concurrent streams")
