"""The split-KV entry point that allocates nothing: fa_fwd_splitkv_static.

Some callers cannot allocate device memory where they run attention -- an
inference engine or plugin host that owns the whole memory budget and gives
out no scratch.  For them the library keeps its own split-KV scratch array
(FA_STATIC_WORKSPACE_BYTES, in device global memory) and this entry point
takes no workspace.  The tests call it through the C ABI and compare it with
the fp64 oracle and with fa_fwd_splitkv (which uses a caller-provided
workspace) on the same inputs, on two calls in a row: the second call finds
the array as the first one left it.  This file is collected last so that a
run stopping at the first failure has already run every other test.
"""

from __future__ import annotations

import numpy as np
import pytest

import exact_tiled_attention_09_gb300 as fa
from fa_inputs import bf16_bits_to_float32, make_custom
from tests.gpu_util import check_parity, from_device, oracle_forward, to_device


def test_static_entry_rejects_sizes_beyond_its_array():
    # 2.2 GB of partials would be needed: refused before any CUDA call
    B, H, L, d, S = 1, 64, 8192, 128, 8
    assert fa.fa_splitkv_workspace_bytes(B, H, L, d, S) > fa.FA_STATIC_WORKSPACE_BYTES
    rc = fa.fa_fwd_splitkv_static(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, B, H, L, d,
                                  0.1, 0, S, None)
    assert rc == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv_static(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 1, 1, 128,
                                    64, 0.1, 0, 0, None) == fa.FA_ERR_INVALID_ARG


def test_scratch_size_follows_the_splits_actually_used():
    # 64 splits requested over 8 key blocks: 8 are used, and the size (which
    # the static entry point checks against its array) is that of 8
    B, H, L, d = 1, 2, 1000, 128
    assert fa.fa_splitkv_workspace_bytes(B, H, L, d, 64) == fa.fa_splitkv_workspace_bytes(
        B, H, L, d, 8)
    assert fa.fa_splitkv_workspace_bytes(B, H, L, d, 64) <= fa.FA_STATIC_WORKSPACE_BYTES
    # 7 splits over 8 blocks take 2 blocks each: 4 splits
    assert fa.fa_splitkv_workspace_bytes(B, H, L, d, 7) == fa.fa_splitkv_workspace_bytes(
        B, H, L, d, 4)


@pytest.mark.gpu
def test_static_entry_matches_workspace_entry_on_two_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    fa.fa_device_status(None, clear=True)
    cases = [  # (B, H, L, d, causal, n_splits, seed): larger first, then smaller
        (1, 2, 1000, 128, 1, 4, 11),
        (2, 3, 700, 64, 0, 3, 12),
        # 64 splits asked for over 8 key blocks: 8 used (64 would not fit)
        (1, 2, 1000, 128, 0, 64, 13),
    ]
    for B, H, L, d, causal, S, seed in cases:
        assert fa.fa_splitkv_workspace_bytes(B, H, L, d, S) <= fa.FA_STATIC_WORKSPACE_BYTES
        qb, kb, vb = make_custom(B, H, L, d, seed=seed)
        q, k, v = (to_device(x, dev) for x in (qb, kb, vb))
        scale = 1.0 / np.sqrt(d)
        o_ws, lse_ws = fa.forward_splitkv(q, k, v, S, scale=scale, causal=bool(causal))
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, L), float("nan"), device=dev)
        stream = torch.cuda.current_stream(dev)
        rc = fa.fa_fwd_splitkv_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), B, H, L, d, float(scale), causal, S,
                                      stream.cuda_stream)
        assert rc == fa.FA_OK, fa.fa_status_string(rc)
        torch.cuda.synchronize()
        a = from_device(o)
        assert np.isfinite(a).all()
        # against the entry point with a caller workspace: the same kernels on
        # the same inputs, only the scratch differs, so the bits agree
        assert bool((o.view(torch.int16) == o_ws.view(torch.int16)).all())
        assert bool((lse == lse_ws).all())
        # against the fp64 oracle on the same inputs
        f = lambda x: bf16_bits_to_float32(x).astype(np.float64)
        o_ref, lse_ref, a_ref = oracle_forward(f(qb), f(kb), f(vb), scale, bool(causal))
        check_parity(a, lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                     f"static split-KV B={B} H={H} L={L} d={d} causal={causal} S={S}", absv_ref=a_ref)
    assert fa.fa_device_status(None, clear=True) == fa.FA_OK
