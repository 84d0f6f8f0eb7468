"""The C ABI boundary, on the host: symbols, status strings, validation.

No test here launches a kernel.  Validation errors are returned before any
CUDA call; the one case with well-formed arguments runs only where no GPU is
present (it must then report FA_ERR_DEVICE).
"""

from __future__ import annotations

import ctypes
import os
import re

import pytest

import exact_tiled_attention_09_gb300 as fa
from exact_tiled_attention_09_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return fa.library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(fa_[a-z_0-9]+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("fa_fwd", "fa_status_string", "fa_device_status", "fa_set_wait_timeout_ns",
              "fa_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(7):
        s = fa.fa_status_string(code)
        assert isinstance(s, str) and s
    assert fa.fa_status_string(0) == "ok"
    assert fa.fa_status_string(99) == "unknown status"
    assert fa.fa_version() >= 100


GOOD = dict(q=0x10000, k=0x20000, v=0x30000, o=0x40000, lse=0x50000,
            B=1, H=1, L=128, d=64, scale=0.125, causal=0)


def _call(**over):
    a = dict(GOOD)
    a.update(over)
    return fa.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["L"],
                     a["d"], a["scale"], a["causal"], None)


@pytest.mark.parametrize("over,code", [
    (dict(q=0), fa.FA_ERR_INVALID_ARG),
    (dict(k=0), fa.FA_ERR_INVALID_ARG),
    (dict(v=0), fa.FA_ERR_INVALID_ARG),
    (dict(o=0), fa.FA_ERR_INVALID_ARG),
    (dict(lse=0), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=-1), fa.FA_ERR_INVALID_ARG),
    (dict(L=0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(B=1 << 16, H=1 << 16), fa.FA_ERR_INVALID_ARG),
    (dict(d=32), fa.FA_ERR_UNSUPPORTED_D),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED_D),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED_D),
    (dict(q=0x10008), fa.FA_ERR_MISALIGNED),
    (dict(o=0x40004), fa.FA_ERR_MISALIGNED),
    (dict(lse=0x50002), fa.FA_ERR_MISALIGNED),
])
def test_validation_errors_launch_nothing(lib, over, code):
    assert _call(**over) == code


def test_well_formed_call_without_gpu_reports_device_error(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; fake pointers must not reach a launch")
    assert _call() == fa.FA_ERR_DEVICE
    assert _call(d=128, causal=1) == fa.FA_ERR_DEVICE


def test_python_forward_rejects_bad_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.forward(q, q, q)  # CPU tensors
    with pytest.raises(ValueError):
        fa.forward(q, q[:, :, :4], q)


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "exact_tiled_attention_09_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src, f


def test_splitkv_workspace_bytes(lib):
    B, H, L, d, S = 2, 3, 300, 64, 5
    rows = B * H * L
    used = 3  # five splits asked for over ceil(300 / 128) = 3 key blocks
    o_bytes = used * rows * d * 4
    expect = ((o_bytes + 255) // 256) * 256 + used * rows * 4
    assert fa.fa_splitkv_workspace_bytes(B, H, L, d, S) == expect
    S2, L2 = 2, 1000  # two splits over 8 blocks: both used
    expect2 = ((S2 * B * H * L2 * d * 4 + 255) // 256) * 256 + S2 * B * H * L2 * 4
    assert fa.fa_splitkv_workspace_bytes(B, H, L2, d, S2) == expect2
    assert fa.fa_splitkv_workspace_bytes(B, H, L, 96, S) == 0
    assert fa.fa_splitkv_workspace_bytes(B, H, L, d, 0) == 0
    assert fa.fa_splitkv_workspace_bytes(B, H, L, d, 65) == 0
    assert fa.fa_splitkv_workspace_bytes(0, H, L, d, S) == 0


def test_splitkv_recommended_splits(lib):
    # as many splits as keep the single-pass CTAs (one per 256 rows of a
    # head) within one wave of 152 SMs, two waves when causal; capped by the
    # number of 128-key blocks and 64; host arithmetic only when the SM count
    # is given
    sms = 152
    assert fa.fa_splitkv_splits(1, 1, 8192, 128, False, sms) == 4     # 32 CTAs
    assert fa.fa_splitkv_splits(1, 1, 16384, 64, False, sms) == 2     # 64 CTAs
    assert fa.fa_splitkv_splits(1, 1, 32768, 128, True, sms) == 2     # 128 CTAs, causal
    assert fa.fa_splitkv_splits(2, 4, 4096, 64, False, sms) == 1      # 128 CTAs
    assert fa.fa_splitkv_splits(1, 8, 8192, 128, True, sms) == 1      # 256 CTAs, causal
    assert fa.fa_splitkv_splits(1, 1, 1024, 64, False, sms) == 8      # 4 CTAs: 8 key blocks
    assert fa.fa_splitkv_splits(1, 1, 128, 64, False, sms) == 1       # one key block
    assert fa.fa_splitkv_splits(1, 1, 100000, 64, False, 1 << 20) == 64  # the cap
    assert fa.fa_splitkv_splits(0, 1, 128, 64, False, sms) == 0
    assert fa.fa_splitkv_splits(1, 1, 128, 96, False, sms) == 0
    assert lib.fa_splitkv_splits(1, 1, 128, 64, 2, sms) == 0


def _call_split(ws=0x1000000, ws_bytes=None, n_splits=4, **over):
    a = dict(GOOD)
    a.update(over)
    if ws_bytes is None:
        ws_bytes = fa.fa_splitkv_workspace_bytes(a["B"], a["H"], a["L"], a["d"], max(1, n_splits))
    return fa.fa_fwd_splitkv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["L"],
                             a["d"], a["scale"], a["causal"], n_splits, ws, ws_bytes, None)


def test_splitkv_validation_launches_nothing(lib):
    assert _call_split(n_splits=0, ws_bytes=1 << 30) == fa.FA_ERR_INVALID_ARG
    assert _call_split(n_splits=65, ws_bytes=1 << 30) == fa.FA_ERR_INVALID_ARG
    assert _call_split(ws=0) == fa.FA_ERR_INVALID_ARG
    assert _call_split(ws_bytes=100) == fa.FA_ERR_INVALID_ARG
    assert _call_split(ws=0x1000010) == fa.FA_ERR_MISALIGNED
    assert _call_split(q=0) == fa.FA_ERR_INVALID_ARG
    assert _call_split(d=96) == fa.FA_ERR_UNSUPPORTED_D
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert _call_split() == fa.FA_ERR_DEVICE


# ---------------------------------------------------------------- backward
BWD_GOOD = dict(q=0x10000, k=0x20000, v=0x30000, o=0x40000, dout=0x50000, lse=0x60000,
                dq=0x70000, dk=0x80000, dv=0x90000, B=1, H=2, L=300, d=64, scale=0.125,
                causal=0, ws=0x1000000)


def test_bwd_workspace_bytes(lib):
    B, H, L, d = 2, 3, 300, 128
    Lp = 384
    acc = ((B * H * L * d * 4 + 255) // 256) * 256
    row = ((B * H * Lp * 4 + 255) // 256) * 256
    sched = 256  # the gradient kernel's unit counter
    assert fa.fa_bwd_workspace_bytes(B, H, L, d) == acc + 2 * row + sched
    assert fa.fa_bwd_workspace_bytes(B, H, L, 96) == 0
    assert fa.fa_bwd_workspace_bytes(0, H, L, d) == 0
    assert fa.fa_bwd_workspace_bytes(B, H, 0, d) == 0


def _call_bwd(ws_bytes=None, **over):
    a = dict(BWD_GOOD)
    a.update(over)
    if ws_bytes is None:
        ws_bytes = fa.fa_bwd_workspace_bytes(a["B"], a["H"], a["L"], a["d"]) or (1 << 30)
    return fa.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["dout"], a["lse"], a["dq"], a["dk"],
                     a["dv"], a["B"], a["H"], a["L"], a["d"], a["scale"], a["causal"], a["ws"],
                     ws_bytes, None)


@pytest.mark.parametrize("over,code", [
    (dict(q=0), fa.FA_ERR_INVALID_ARG),
    (dict(o=0), fa.FA_ERR_INVALID_ARG),
    (dict(dout=0), fa.FA_ERR_INVALID_ARG),
    (dict(lse=0), fa.FA_ERR_INVALID_ARG),
    (dict(dq=0), fa.FA_ERR_INVALID_ARG),
    (dict(dk=0), fa.FA_ERR_INVALID_ARG),
    (dict(dv=0), fa.FA_ERR_INVALID_ARG),
    (dict(ws=0), fa.FA_ERR_INVALID_ARG),
    (dict(ws_bytes=1000), fa.FA_ERR_INVALID_ARG),
    (dict(L=0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=3), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(B=1 << 16, H=1 << 16), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED_D),
    (dict(dout=0x50008), fa.FA_ERR_MISALIGNED),
    (dict(dk=0x80002), fa.FA_ERR_MISALIGNED),
    (dict(lse=0x60002), fa.FA_ERR_MISALIGNED),
    (dict(ws=0x1000080), fa.FA_ERR_MISALIGNED),
])
def test_bwd_validation_errors_launch_nothing(lib, over, code):
    assert _call_bwd(**over) == code


def test_bwd_well_formed_call_without_gpu_reports_device_error(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; fake pointers must not reach a launch")
    assert _call_bwd() == fa.FA_ERR_DEVICE
    assert _call_bwd(d=128, causal=1) == fa.FA_ERR_DEVICE


def test_python_backward_rejects_bad_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 1, 8)
    with pytest.raises(ValueError):
        fa.backward(q, q, q, q, lse, q)  # CPU tensors


# ---------------------------------------------------------------- FP8
def test_fp8_validation_launches_nothing(lib):
    q = dict(x=0x10000, codes=0x20000, scales=0x30000)
    call_q = lambda **o: fa.fa_quantize_fp8(o.get("x", q["x"]), o.get("codes", q["codes"]),
                                            o.get("scales", q["scales"]), 1, 2, o.get("L", 300),
                                            o.get("d", 64), None)
    assert call_q(x=0) == fa.FA_ERR_INVALID_ARG
    assert call_q(L=0) == fa.FA_ERR_INVALID_ARG
    assert call_q(d=96) == fa.FA_ERR_UNSUPPORTED_D
    assert call_q(codes=0x20008) == fa.FA_ERR_MISALIGNED
    assert call_q(scales=0x30002) == fa.FA_ERR_MISALIGNED
    f = lambda qs=0x40000, ks=0x50000, **o: fa.fa_fwd_fp8(
        o.get("q8", 0x10000), 0x20000, 0x30000, qs, ks, 0x60000, 0x70000, 1, 2,
        o.get("L", 300), o.get("d", 128), 0.1, 0, None)
    assert f(qs=0) == fa.FA_ERR_INVALID_ARG
    assert f(ks=0) == fa.FA_ERR_INVALID_ARG
    assert f(qs=0x40002) == fa.FA_ERR_MISALIGNED
    assert f(q8=0) == fa.FA_ERR_INVALID_ARG
    assert f(d=32) == fa.FA_ERR_UNSUPPORTED_D
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert call_q() == fa.FA_ERR_DEVICE
        assert f() == fa.FA_ERR_DEVICE


def test_host_forward_validation_launches_nothing(lib):
    n = fa.fa_fwd_host_workspace_bytes(1, 2, 300, 64)
    assert n == ((4 * 1 * 2 * 300 * 64 * 2 + 255) // 256) * 256 + 1 * 2 * 300 * 4
    assert fa.fa_fwd_host_workspace_bytes(1, 2, 300, 96) == 0
    call = lambda ws=0x1000000, wsb=n, **o: fa.fa_fwd_host(
        o.get("q", 0x10000), 0x20000, 0x30000, 0x40000, 0x50000, 1, 2, o.get("L", 300),
        o.get("d", 64), 0.125, 0, ws, wsb, None)
    assert call(q=0) == fa.FA_ERR_INVALID_ARG
    assert call(ws=0) == fa.FA_ERR_INVALID_ARG
    assert call(wsb=n - 1) == fa.FA_ERR_INVALID_ARG
    assert call(ws=0x1000010) == fa.FA_ERR_MISALIGNED
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED_D
    assert call(L=0) == fa.FA_ERR_INVALID_ARG
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert call() == fa.FA_ERR_DEVICE
