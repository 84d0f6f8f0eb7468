"""GPU tests of fa_fwd_host: the forward on host buffers (copies in, kernel,
copies out on one stream), through the C ABI.

Its outputs must equal the device-buffer forward bit for bit (the same
kernel on the same values), with the inputs packed back to back in host
memory (one copy) or apart (three copies), and calls pipelined over two
streams with two workspaces must each produce their own step's result.
"""

from __future__ import annotations

import numpy as np
import pytest

import exact_tiled_attention_09_gb300 as fa
from fa_inputs import bf16_bits_to_float32, make_custom
from tests.gpu_util import check_parity, oracle_forward, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.library()
    yield torch.device("cuda:0")
    assert fa.fa_device_status(None, clear=True) == fa.FA_OK


def _host(bits, pinned=True):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pinned else t


@pytest.mark.parametrize("packed", [True, False])
@pytest.mark.parametrize("d,causal", [(64, False), (128, True)])
def test_host_forward_equals_device_forward(dev, packed, d, causal):
    import torch
    B, H, L = 2, 3, 333
    qb, kb, vb = make_custom(B, H, L, d, 5000 + d)
    if packed:
        buf = _host(np.concatenate([qb.ravel(), kb.ravel(), vb.ravel()]))
        n = qb.size
        q, k, v = (buf[i * n:(i + 1) * n].view(B, H, L, d) for i in range(3))
        out_buf = torch.empty(n * 2 + B * H * L * 4, dtype=torch.uint8).pin_memory()
        o = out_buf[:n * 2].view(torch.bfloat16).view(B, H, L, d)
        lse = out_buf[n * 2:].view(torch.float32).view(B, H, L)
    else:
        q, k, v = (_host(x) for x in (qb, kb, vb))
        o = torch.empty_like(q).pin_memory()
        lse = torch.empty((B, H, L), dtype=torch.float32).pin_memory()
    fa.forward_host(q, k, v, scale=0.1, causal=causal, out=o, lse=lse, device=dev)
    torch.cuda.synchronize()
    od, ld = fa.forward(*(to_device(x, dev) for x in (qb, kb, vb)), scale=0.1, causal=causal)
    torch.cuda.synchronize()
    assert bool((o.view(torch.int16) == od.cpu().view(torch.int16)).all())
    assert bool((lse == ld.cpu()).all())
    f = lambda b: bf16_bits_to_float32(b).astype(np.float64)
    o_ref, lse_ref, a_ref = oracle_forward(f(qb), f(kb), f(vb), 0.1, causal)
    check_parity(o.float().numpy().astype(np.float64), lse.numpy().astype(np.float64), o_ref,
                 lse_ref, f"host packed={packed}", absv_ref=a_ref)


def test_host_forward_pipelined_on_two_streams(dev):
    import torch
    B, H, L, d = 1, 4, 700, 64
    inputs = [make_custom(B, H, L, d, 5100 + i) for i in range(4)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    need = fa.fa_fwd_host_workspace_bytes(B, H, L, d)
    ws = [torch.empty(need, dtype=torch.uint8, device=dev) for _ in range(2)]
    hosts = [[_host(x) for x in inp] for inp in inputs]
    outs = [(torch.empty((B, H, L, d), dtype=torch.bfloat16).pin_memory(),
             torch.empty((B, H, L), dtype=torch.float32).pin_memory()) for _ in inputs]
    for i, (hq, hk, hv) in enumerate(hosts):
        fa.forward_host(hq, hk, hv, causal=True, out=outs[i][0], lse=outs[i][1],
                        workspace=ws[i % 2], stream=streams[i % 2], device=dev)
    torch.cuda.synchronize()
    for i, (qb, kb, vb) in enumerate(inputs):
        od, ld = fa.forward(*(to_device(x, dev) for x in (qb, kb, vb)), causal=True)
        torch.cuda.synchronize()
        assert bool((outs[i][0].view(torch.int16) == od.cpu().view(torch.int16)).all()), i
        assert bool((outs[i][1] == ld.cpu()).all()), i
