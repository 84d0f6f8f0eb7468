"""Failure detection without a GPU fault: a kernel wait that runs out.

Every mbarrier wait in the kernels is bounded in time.  With the test hook
fa_test_withhold_q_load the producer skips its Q copy, so the MMA warp's
first wait never completes.  After the (shortened) wait limit the kernel
must record the timeout, stop every role, drain its own copies, free its
tensor memory and return.  The host then reads FA_ERR_TIMEOUT from
fa_device_status, and the CUDA context stays usable: a normal forward right
after it matches the oracle.  Nothing here traps, asserts on the device or
hangs.
"""

from __future__ import annotations

import math
import time

import numpy as np
import pytest

import exact_tiled_attention_09_gb300 as fa
import oracle
from fa_inputs import bf16_bits_to_float32, make_custom
from tests.gpu_util import check_parity, oracle_forward, from_device, to_device

pytestmark = pytest.mark.gpu

SHORT_LIMIT_NS = 20_000_000        # 20 ms
DEFAULT_LIMIT_NS = 1_000_000_000   # the library default


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.library()
    fa.fa_device_status(None, clear=True)
    yield torch.device("cuda:0")
    fa.fa_test_withhold_q_load(False)
    fa.fa_set_wait_timeout_ns(DEFAULT_LIMIT_NS)
    fa.fa_device_status(None, clear=True)


def _f64(bits):
    return bf16_bits_to_float32(bits).astype(np.float64)


@pytest.mark.parametrize("d,causal,split", [(64, False, 0), (64, True, 3), (128, True, 0),
                                           (128, False, 3)])
def test_wait_that_runs_out_is_reported_and_the_context_survives(dev, d, causal, split):
    import torch
    B, H, L = 2, 3, 600
    qb, kb, vb = make_custom(B, H, L, d, seed=700 + d + split)
    q, k, v = (to_device(x, dev) for x in (qb, kb, vb))
    scale = 1.0 / math.sqrt(d)
    run = (lambda: fa.forward_splitkv(q, k, v, split, scale=scale, causal=causal)) if split \
        else (lambda: fa.forward(q, k, v, scale=scale, causal=causal))

    assert fa.fa_device_status(None, clear=True) == fa.FA_OK
    try:
        fa.fa_set_wait_timeout_ns(SHORT_LIMIT_NS)
        fa.fa_test_withhold_q_load(True)
        t0 = time.time()
        run()  # the launch itself succeeds; the kernel gives up inside
        torch.cuda.synchronize()
        elapsed = time.time() - t0
        status = fa.fa_device_status(None, clear=True)
    finally:
        fa.fa_test_withhold_q_load(False)
        fa.fa_set_wait_timeout_ns(DEFAULT_LIMIT_NS)
    assert status == fa.FA_ERR_TIMEOUT
    assert elapsed < 10.0, f"the withheld wait took {elapsed:.1f} s to end"

    # the same context keeps working
    o, lse = run()
    torch.cuda.synchronize()
    assert fa.fa_device_status(None, clear=True) == fa.FA_OK
    o_ref, lse_ref, a_ref = oracle_forward(_f64(qb), _f64(kb), _f64(vb), scale, causal)
    check_parity(from_device(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                 f"after timeout d={d} causal={causal} split={split}", absv_ref=a_ref)


@pytest.mark.parametrize("d,causal", [(64, False), (64, True), (128, False)])
def test_fp8_wait_that_runs_out_is_reported(dev, d, causal):
    # FP8 at d = 64 runs two MMA warps (one per 128-query tile) and its own
    # code path for the K scales: every role must still stop, drain and return
    import torch
    from tests.test_fp8_gpu import _fp8_case
    B, H, L = 2, 3, 600
    qb, kb, vb = make_custom(B, H, L, d, seed=720 + d + int(causal))
    q, k, v = (to_device(x, dev) for x in (qb, kb, vb))
    scale = 1.0 / math.sqrt(d)
    q8, qs = fa.quantize_fp8(q)
    k8, ks = fa.quantize_fp8(k)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None, clear=True) == fa.FA_OK
    try:
        fa.fa_set_wait_timeout_ns(SHORT_LIMIT_NS)
        fa.fa_test_withhold_q_load(True)
        t0 = time.time()
        fa.forward_fp8(q8, k8, v, qs, ks, scale=scale, causal=causal)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
        status = fa.fa_device_status(None, clear=True)
    finally:
        fa.fa_test_withhold_q_load(False)
        fa.fa_set_wait_timeout_ns(DEFAULT_LIMIT_NS)
    assert status == fa.FA_ERR_TIMEOUT
    assert elapsed < 10.0, f"the withheld wait took {elapsed:.1f} s to end"
    # the same context keeps working: a full FP8 forward against the oracle
    _fp8_case(dev, qb, kb, vb, scale, causal, f"fp8 after timeout d={d} causal={causal}")
    assert fa.fa_device_status(None, clear=True) == fa.FA_OK


@pytest.mark.parametrize("d,causal", [(64, False), (128, True)])
def test_backward_wait_that_runs_out_is_reported(dev, d, causal):
    import torch
    from fa_inputs import make_custom_grad_out
    B, H, L = 1, 2, 300
    qb, kb, vb = make_custom(B, H, L, d, seed=710 + d)
    dob = make_custom_grad_out(B, H, L, d, 710 + d)
    q, k, v, do = (to_device(x, dev) for x in (qb, kb, vb, dob))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.forward(q, k, v, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None, clear=True) == fa.FA_OK
    try:
        fa.fa_set_wait_timeout_ns(SHORT_LIMIT_NS)
        fa.fa_test_withhold_q_load(True)  # the backward kernel skips its K/V copy
        t0 = time.time()
        fa.backward(q, k, v, o, lse, do, scale=scale, causal=causal)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
        status = fa.fa_device_status(None, clear=True)
    finally:
        fa.fa_test_withhold_q_load(False)
        fa.fa_set_wait_timeout_ns(DEFAULT_LIMIT_NS)
    assert status == fa.FA_ERR_TIMEOUT
    assert elapsed < 10.0
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None, clear=True) == fa.FA_OK
    ref = oracle.attention_bwd(_f64(qb), _f64(kb), _f64(vb), _f64(dob), scale, causal)
    from tests.gpu_util import check_grads_per_head
    check_grads_per_head([from_device(t) for t in (dq, dk, dv)], ref, "bwd after timeout")
