"""GB300 (sm_103a) exact attention, forward and backward: Python binding of
``include/fa.h``.

The binding only marshals arguments; every step of the computation runs in
the CUDA kernels of ``libfa_gb300.so``.  PyTorch is used for device memory and
the current stream.  There is no fallback: if the library is missing or the
device is not sm_103, calls raise.

    o, lse = forward(q, k, v, scale=None, causal=False)

q, k, v: CUDA bf16 tensors [B, H, L, d] (contiguous), d in {64, 128}.
Returns o (bf16, same shape) and lse (fp32 [B, H, L], natural log).

    dq, dk, dv = backward(q, k, v, o, lse, do, scale=None, causal=False)

takes the forward's o and lse and the output gradient do (bf16, shaped like
q) and returns the bf16 input gradients.
"""

from __future__ import annotations

import ctypes
import math
import os

from .build import LIB

__all__ = [
    "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED_D", "FA_ERR_MISALIGNED",
    "FA_ERR_DEVICE", "FA_ERR_LAUNCH", "FA_ERR_TIMEOUT", "FAError",
    "library", "fa_fwd", "fa_fwd_splitkv", "fa_fwd_splitkv_static", "FA_STATIC_WORKSPACE_BYTES",
    "fa_splitkv_workspace_bytes", "fa_splitkv_splits", "fa_device_status",
    "fa_set_wait_timeout_ns", "fa_test_withhold_q_load", "fa_status_string", "fa_version",
    "fa_bwd", "fa_bwd_workspace_bytes", "fa_quantize_fp8", "fa_fwd_fp8",
    "fa_fwd_host", "fa_fwd_host_workspace_bytes", "forward_host",
    "forward", "forward_splitkv", "backward", "quantize_fp8", "forward_fp8",
    "flops", "flops_bwd",
]

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED_D = 2
FA_ERR_MISALIGNED = 3
FA_ERR_DEVICE = 4
FA_ERR_LAUNCH = 5
FA_ERR_TIMEOUT = 6


class FAError(RuntimeError):
    def __init__(self, code: int, where: str = "fa_fwd"):
        self.code = code
        super().__init__(f"{where}: {fa_status_string(code)} (status {code})")


_lib = None


def library() -> ctypes.CDLL:
    """The loaded kernel library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(
                f"{LIB} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(this package has no CPU or eager fallback)")
        lib = ctypes.CDLL(LIB)
        vp, ci = ctypes.c_void_p, ctypes.c_int
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ctypes.c_float, ci, vp]
        lib.fa_fwd.restype = ci
        lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ctypes.c_float, ci, ci,
                                       vp, ctypes.c_size_t, vp]
        lib.fa_fwd_splitkv.restype = ci
        lib.fa_fwd_splitkv_static.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ctypes.c_float,
                                              ci, ci, vp]
        lib.fa_fwd_splitkv_static.restype = ci
        lib.fa_splitkv_workspace_bytes.argtypes = [ci, ci, ci, ci, ci]
        lib.fa_splitkv_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_splitkv_splits.argtypes = [ci, ci, ci, ci, ci, ci]
        lib.fa_splitkv_splits.restype = ci
        lib.fa_device_status.argtypes = [vp, ci]
        lib.fa_device_status.restype = ci
        lib.fa_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        lib.fa_set_wait_timeout_ns.restype = None
        lib.fa_test_withhold_q_load.argtypes = [ci]
        lib.fa_test_withhold_q_load.restype = None
        lib.fa_status_string.argtypes = [ci]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci,
                               ctypes.c_float, ci, vp, ctypes.c_size_t, vp]
        lib.fa_bwd.restype = ci
        lib.fa_bwd_workspace_bytes.argtypes = [ci, ci, ci, ci]
        lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_quantize_fp8.argtypes = [vp, vp, vp, ci, ci, ci, ci, vp]
        lib.fa_quantize_fp8.restype = ci
        lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ctypes.c_float, ci,
                                   vp]
        lib.fa_fwd_fp8.restype = ci
        lib.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ctypes.c_float, ci, vp,
                                    ctypes.c_size_t, vp]
        lib.fa_fwd_host.restype = ci
        lib.fa_fwd_host_workspace_bytes.argtypes = [ci, ci, ci, ci]
        lib.fa_fwd_host_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_version.argtypes = []
        lib.fa_version.restype = ci
        _lib = lib
    return _lib


# ---------------------------------------------------------------- raw C ABI
def fa_fwd(q, k, v, o, lse, B, H, L, d, scale, causal, stream) -> int:
    """Direct call of the C entry point with integer device addresses."""
    return library().fa_fwd(q, k, v, o, lse, B, H, L, d, scale, causal, stream)


def fa_fwd_splitkv(q, k, v, o, lse, B, H, L, d, scale, causal, n_splits, workspace,
                   workspace_bytes, stream) -> int:
    """Direct call of the split-KV C entry point with integer addresses."""
    return library().fa_fwd_splitkv(q, k, v, o, lse, B, H, L, d, scale, causal, n_splits,
                                    workspace, workspace_bytes, stream)


def fa_fwd_splitkv_static(q, k, v, o, lse, B, H, L, d, scale, causal, n_splits, stream) -> int:
    """Split-KV on the library's own static scratch array (no workspace, no
    allocation); for callers that cannot allocate device memory."""
    return library().fa_fwd_splitkv_static(q, k, v, o, lse, B, H, L, d, scale, causal,
                                           n_splits, stream)


# Size of the static scratch array behind fa_fwd_splitkv_static (fa.h).
FA_STATIC_WORKSPACE_BYTES = 64 << 20


def fa_splitkv_workspace_bytes(B, H, L, d, n_splits) -> int:
    return library().fa_splitkv_workspace_bytes(B, H, L, d, n_splits)


def fa_splitkv_splits(B, H, L, d, causal, num_sms=0) -> int:
    return library().fa_splitkv_splits(B, H, L, d, int(bool(causal)), num_sms)


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, L, d, scale, causal, workspace,
           workspace_bytes, stream) -> int:
    """Direct call of the backward C entry point with integer addresses."""
    return library().fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, L, d, scale, causal,
                            workspace, workspace_bytes, stream)


def fa_bwd_workspace_bytes(B, H, L, d) -> int:
    return library().fa_bwd_workspace_bytes(B, H, L, d)


def fa_quantize_fp8(x, codes, scales, B, H, L, d, stream) -> int:
    """Direct call of the FP8 block quantisation with integer addresses."""
    return library().fa_quantize_fp8(x, codes, scales, B, H, L, d, stream)


def fa_fwd_fp8(q8, k8, v, q_scale, k_scale, o, lse, B, H, L, d, scale, causal, stream) -> int:
    """Direct call of the FP8 forward with integer addresses."""
    return library().fa_fwd_fp8(q8, k8, v, q_scale, k_scale, o, lse, B, H, L, d, scale, causal,
                                stream)


def fa_fwd_host(q, k, v, o, lse, B, H, L, d, scale, causal, workspace, workspace_bytes,
                stream) -> int:
    """Direct call of the host-buffer forward with integer addresses."""
    return library().fa_fwd_host(q, k, v, o, lse, B, H, L, d, scale, causal, workspace,
                                 workspace_bytes, stream)


def fa_fwd_host_workspace_bytes(B, H, L, d) -> int:
    return library().fa_fwd_host_workspace_bytes(B, H, L, d)


def fa_device_status(stream=None, clear=True) -> int:
    return library().fa_device_status(stream, int(bool(clear)))


def fa_set_wait_timeout_ns(ns: int) -> None:
    library().fa_set_wait_timeout_ns(int(ns))


def fa_test_withhold_q_load(enable: bool) -> None:
    """Test hook of the timeout path (see fa.h); leave disabled otherwise."""
    library().fa_test_withhold_q_load(int(bool(enable)))


def fa_status_string(code: int) -> str:
    return library().fa_status_string(int(code)).decode()


def fa_version() -> int:
    return library().fa_version()


# ---------------------------------------------------------------- torch API
def flops(B, H, L, d, causal) -> float:
    """Forward FLOPs by the metric's convention: 4*B*H*L^2*d, halved if causal."""
    f = 4.0 * B * H * L * L * d
    return f / 2 if causal else f


def flops_bwd(B, H, L, d, causal) -> float:
    """Backward FLOPs by the usual convention: five L x L x d products,
    10*B*H*L^2*d (2.5 x the forward), halved if causal."""
    f = 10.0 * B * H * L * L * d
    return f / 2 if causal else f


def forward(q, k, v, scale=None, causal=False, out=None, lse=None, stream=None):
    """Exact attention forward on CUDA bf16 tensors [B, H, L, d].

    ``scale`` defaults to 1/sqrt(d).  ``out``/``lse`` may be preallocated.
    Launches asynchronously on ``stream`` (default: torch's current stream).
    """
    import torch

    if q.shape != k.shape or q.shape != v.shape or q.dim() != 4:
        raise ValueError("q, k, v must share one shape [B, H, L, d]")
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA bfloat16 tensors")
    B, H, L, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if lse.shape != (B, H, L) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, H, L]")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        rc = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                    B, H, L, d, float(scale), int(bool(causal)), stream.cuda_stream)
    if rc != FA_OK:
        raise FAError(rc)
    return out, lse


def forward_splitkv(q, k, v, n_splits=None, scale=None, causal=False, out=None, lse=None,
                    workspace=None, stream=None):
    """:func:`forward` computed in ``n_splits`` key splits plus a merge
    (``None``: the library's recommendation, ``fa_splitkv_splits``).

    ``workspace`` (a CUDA uint8 tensor of at least
    ``fa_splitkv_workspace_bytes(B, H, L, d, n_splits)`` bytes, 256-byte
    aligned) is allocated here when not given.
    """
    import torch

    if q.shape != k.shape or q.shape != v.shape or q.dim() != 4:
        raise ValueError("q, k, v must share one shape [B, H, L, d]")
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA bfloat16 tensors")
    B, H, L, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if n_splits is None:
        with torch.cuda.device(q.device):
            n_splits = fa_splitkv_splits(B, H, L, d, causal)
    need = fa_splitkv_workspace_bytes(B, H, L, d, n_splits)
    if need == 0:
        raise ValueError("invalid sizes or n_splits for split-KV")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        rc = fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            lse.data_ptr(), B, H, L, d, float(scale), int(bool(causal)),
                            int(n_splits), workspace.data_ptr(),
                            workspace.numel() * workspace.element_size(), stream.cuda_stream)
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_splitkv")
    return out, lse


def backward(q, k, v, o, lse, do, scale=None, causal=False, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """Gradients of exact attention: returns (dq, dk, dv), bf16 like q.

    q, k, v, o, do: contiguous CUDA bf16 [B, H, L, d]; lse: fp32 [B, H, L]
    from :func:`forward` with the same ``scale`` and ``causal``.
    ``workspace`` (CUDA uint8, >= ``fa_bwd_workspace_bytes(B, H, L, d)``
    bytes, 256-byte aligned) is allocated here when not given.
    """
    import torch

    if not (q.shape == k.shape == v.shape == o.shape == do.shape) or q.dim() != 4:
        raise ValueError("q, k, v, o, do must share one shape [B, H, L, d]")
    for t in (q, k, v, o, do):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v, o, do must be contiguous CUDA bfloat16 tensors")
    B, H, L, d = q.shape
    if lse.shape != (B, H, L) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, H, L]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = fa_bwd_workspace_bytes(B, H, L, d)
    if need == 0:
        raise ValueError("invalid sizes for the backward pass")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for t in (dq, dk, dv):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("dq, dk, dv must be contiguous bf16 tensors shaped like q")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        rc = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                    lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, L, d,
                    float(scale), int(bool(causal)), workspace.data_ptr(),
                    workspace.numel() * workspace.element_size(), stream.cuda_stream)
    if rc != FA_OK:
        raise FAError(rc, "fa_bwd")
    return dq, dk, dv


def quantize_fp8(x, codes=None, scales=None, stream=None):
    """E4M3 block quantisation of a CUDA bf16 tensor [B, H, L, d]: returns
    (codes uint8 [B, H, L, d], scales fp32 [B, H, ceil(L/128)])."""
    import torch

    if x.dim() != 4 or x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA bf16 tensor [B, H, L, d]")
    B, H, L, d = x.shape
    nb = (L + 127) // 128
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((B, H, nb), dtype=torch.float32, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    with torch.cuda.device(x.device):
        rc = fa_quantize_fp8(x.data_ptr(), codes.data_ptr(), scales.data_ptr(), B, H, L, d,
                             stream.cuda_stream)
    if rc != FA_OK:
        raise FAError(rc, "fa_quantize_fp8")
    return codes, scales


def forward_fp8(q8, k8, v, q_scale, k_scale, scale=None, causal=False, out=None, lse=None,
                stream=None):
    """Attention forward with E4M3 Q and K (codes and block scales from
    :func:`quantize_fp8`) and bf16 V; returns (o bf16, lse fp32)."""
    import torch

    if q8.shape != k8.shape or q8.shape != v.shape or q8.dim() != 4:
        raise ValueError("q8, k8, v must share one shape [B, H, L, d]")
    if q8.dtype != torch.uint8 or k8.dtype != torch.uint8 or v.dtype != torch.bfloat16:
        raise ValueError("q8, k8 must be uint8 codes and v bf16")
    for t in (q8, k8, v, q_scale, k_scale):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    B, H, L, d = v.shape
    nb = (L + 127) // 128
    for t in (q_scale, k_scale):
        if t.shape != (B, H, nb) or t.dtype != torch.float32:
            raise ValueError("scales must be fp32 [B, H, ceil(L/128)]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(v)
    if lse is None:
        lse = torch.empty((B, H, L), dtype=torch.float32, device=v.device)
    if stream is None:
        stream = torch.cuda.current_stream(v.device)
    with torch.cuda.device(v.device):
        rc = fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v.data_ptr(), q_scale.data_ptr(),
                        k_scale.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, L, d,
                        float(scale), int(bool(causal)), stream.cuda_stream)
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_fp8")
    return out, lse


def forward_host(q, k, v, scale=None, causal=False, out=None, lse=None, workspace=None,
                 stream=None, device=None):
    """:func:`forward` on CPU tensors: copies in, forward, copies out, all on
    ``stream`` (asynchronous when the tensors are pinned; synchronise the
    stream before reading ``out``/``lse``).  ``workspace`` is a CUDA uint8
    tensor of at least ``fa_fwd_host_workspace_bytes`` bytes."""
    import torch

    if q.shape != k.shape or q.shape != v.shape or q.dim() != 4:
        raise ValueError("q, k, v must share one shape [B, H, L, d]")
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CPU bfloat16 tensors")
    B, H, L, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    device = device or torch.device("cuda", torch.cuda.current_device())
    need = fa_fwd_host_workspace_bytes(B, H, L, d)
    if need == 0:
        raise ValueError("invalid sizes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, L), dtype=torch.float32)
    if stream is None:
        stream = torch.cuda.current_stream(device)
    with torch.cuda.device(device):
        rc = fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                         B, H, L, d, float(scale), int(bool(causal)), workspace.data_ptr(),
                         workspace.numel() * workspace.element_size(), stream.cuda_stream)
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_host")
    return out, lse
