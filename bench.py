"""Benchmark: exact attention forward TFLOPS on GB300 (one JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one attention forward (the whole hot path, one kernel launch) over
the headline workload B=1, H=16, L=32768, d=64, non-causal, scale 1/8, inputs
Q, K, V ~ N(0,1) drawn by the seeded generator and rounded to bf16: the
largest of the synthetic configurations, 4.4e12 FLOP per launch.  The inputs
are resident in HBM when timing starts; L2 is flushed (a 512 MiB write)
before every timed step, outside the timed events.

FLOPs per step follow the metric: 4*B*H*L^2*d (halved when causal).
``value`` = whole-job TFLOP/s = N * FLOPs * K / max over ranks of the summed
device time of K steps (CUDA events on the launching stream).
``e2e`` = the same metric through the public host-buffer call
(``fa_fwd_host``) with pinned host buffers: every step copies Q, K, V
host->device, runs the forward and copies O and LSE back, all inside the
timed region; steps alternate two workspaces on two streams so one step's
copies overlap the previous step (the serial figure is reported beside it).
``roofline`` compares the kernel against the measured dense bf16 peak.
``cpu_baseline`` times the fp64 oracle on the host cores on a bounded sample
of the same inputs, after the GPU timing.
``splitkv`` times the split-KV path (split pass + merge) against the single
pass on shapes whose single-pass grid underfills the GPU.  ``backward`` times
the backward pass (gradients by recomputation) on every workload: TFLOP/s by
the convention 10*B*H*L^2*d (five L x L x d products; halved when causal).
``fp8`` times the FP8 forward (E4M3 Q and K with block scales, bf16 V) on
every workload by the forward's convention, against the dense FP8 ceiling
(the measured bf16 peak times the nominal fp8/bf16 rate ratio of 2), and the
block quantisation of Q and K apart.  ``workloads`` (the last key) lists the
bf16 forward on every synthetic configuration (device-generated seeded
inputs), each timed the same way, including the d=128 non-causal L=8192 point
used for the tensor-core fraction.

With more than one GPU (torchrun) every rank runs its own replica of the
workload (the forward pass has no exchange step); only the timing is
reduced (max over ranks).

``--impl reference`` times the fp64 CPU oracle instead (rank 0 only): each
step is one oracle pass over a bounded sample of rows of the headline
workload.
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADLINE = "B1_H16_L32768_d64"
METRIC = "attention fwd TFLOPS (4·B·H·L²·d) and % of GB300 dense BF16 tensor peak"
FLUSH_BYTES = 512 << 20
# NVIDIA's nominal dense bf16 tensor rate for one GB300, 2.25 PFLOP/s (its
# published 2:4-sparse figure halved).  Reported as a second denominator next
# to the measured peak; the roofline fractions use the measured one.
NOMINAL_BF16_TFLOPS = 2250.0
# Dense FP8 (E4M3) runs at twice the dense bf16 rate on this tensor core
# (nominal 4.5 against 2.25 PFLOP/s); the FP8 ceiling is the measured bf16
# peak scaled by that ratio.
FP8_OVER_BF16 = 2.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- helpers
def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# Device-code files each kernel is built from; a profile summary records the
# hash of these files at capture time and is used only while it matches.
KERNEL_SOURCES = {
    "fwd": ["fa_fwd_kernel.cuh", "sm103_ptx.cuh"],
    "fwd_fp8": ["fa_fwd_kernel.cuh", "sm103_ptx.cuh"],
    "bwd": ["fa_bwd_kernel.cuh", "sm103_ptx.cuh"],
}


def _code_only(src: str) -> str:
    """C++ source with comments removed and whitespace runs collapsed, so that
    editing a comment does not change the kernel's source hash.  String and
    character literals (the inline PTX) are kept verbatim."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(kernel: str = "fwd") -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "exact_tiled_attention_09_gb300", "csrc", name),
                  encoding="utf-8") as fh:
            h.update(name.encode())
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def read_traffic(workload: str, kernel: str = "fwd"):
    """DRAM bytes per launch from the committed ncu summary of this kernel on
    this workload, if it was captured on the current kernel source; else None."""
    src = kernel_source_hash(kernel)
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        text = open(path).read()
        m_k = re.search(r"^kernel:\s*(\S+)", text, re.M)
        m_w = re.search(r"^workload:\s*(\S+)", text, re.M)
        m_h = re.search(r"^kernel_source_sha256_16:\s*(\S+)", text, re.M)
        m_t = re.search(r"^dram_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
        k = m_k.group(1) if m_k else "fwd"
        if (k == kernel and m_w and m_h and m_t and m_w.group(1) == workload
                and m_h.group(1) == src):
            return float(m_t.group(1)), os.path.relpath(path, ROOT)
    return None, None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU works."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"fa_bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[4:9], float(parts[3])))
            except ValueError:
                continue
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm_max = max(r[1] for r in rows)
        loaded = [r for r in rows if r[3] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i in range(4)
                          if r[2][1 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": sm_max,
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r[3] for r in rows)}


# ----------------------------------------------------------------- CPU leg
def row_flops(w, rows):
    """Work of the given query rows of one head under the metric's convention:
    4*L*d per row (non-causal); causal rows count their visible keys, 4*(i+1)*d
    for row i (a whole head then sums to 2*L*(L+1)*d, the halved count up to
    the diagonal)."""
    import numpy as np
    rows = np.asarray(rows, dtype=np.int64)
    if w.causal:
        return 4.0 * w.d * float((rows + 1).sum())
    return 4.0 * w.L * w.d * rows.size


def oracle_sample_run(w, qb, kb, vb, heads, n_rows, threads=0):
    """One oracle pass over the first ``n_rows`` query rows of each of the
    first ``heads`` heads of the workload (every key of those heads);
    returns (seconds, flops)."""
    import numpy as np

    import oracle
    from fa_inputs import bf16_bits_to_float32

    BH = w.B * w.H
    f = lambda b: bf16_bits_to_float32(b.reshape(BH, w.L, w.d)[:heads]).astype(np.float64)
    q, k, v = f(qb), f(kb), f(vb)
    rows = None if n_rows >= w.L else [h * w.L + i for h in range(heads) for i in range(n_rows)]
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.scale, w.causal, rows=rows, threads=threads)
    dt = time.perf_counter() - t0
    return dt, heads * row_flops(w, range(min(n_rows, w.L)))


def sample_size(w, qb, kb, vb, target_s):
    """(heads, rows per head) of a sample taking about ``target_s`` seconds:
    rows of the first head while one head is more than enough, else whole
    heads.  Sized from a probe of 256 rows."""
    probe = min(256, w.L)
    dt, _ = oracle_sample_run(w, qb, kb, vb, 1, probe)
    per_row = max(dt, 1e-6) / probe
    rows = int(target_s / per_row)
    if rows < w.L:
        return 1, max(1, rows)
    return max(1, min(w.B * w.H, int(target_s / (per_row * w.L)))), w.L


def cpu_baseline(w, qb, kb, vb, target_s=8.0):
    """Oracle TFLOP/s on the host cores, on a bounded sample of the workload."""
    BH = w.B * w.H
    heads, rows = sample_size(w, qb, kb, vb, target_s)
    dt, fl = oracle_sample_run(w, qb, kb, vb, heads, rows)
    cores = os.cpu_count() or 1
    what = (f"query rows 0..{rows - 1} of head 0" if heads == 1 and rows < w.L
            else f"{heads} of {BH} whole heads")
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{what} of {w.name} (every key), fp64, {dt:.1f} s wall, "
                      f"{cores} threads, after the GPU timing"}


def step_stats(t):
    """Mean, median, 90th percentile and minimum of per-step times (ms)."""
    s = sorted(t)
    p90 = s[min(len(s) - 1, int(math.ceil(0.9 * len(s))) - 1)]
    return {"ms_mean": round(sum(s) / len(s), 5), "ms_median": round(statistics.median(s), 5),
            "ms_p90": round(p90, 5), "ms_min": round(s[0], 5)}


# ----------------------------------------------------------------- GPU leg
def device_inputs(w, dev, torch):
    """Seeded normal inputs generated on the device (for the extra workloads)."""
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    shape = (w.B, w.H, w.L, w.d)
    mk = lambda s: (torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * s).to(
        torch.bfloat16)
    return mk(w.q_std), mk(w.k_std), mk(w.v_std)


def time_forward(fa, torch, q, k, v, w, steps, warmup, flush_buf, o=None, lse=None):
    """Per-step device time (ms) of ``fa.forward``; L2 flushed before each step."""
    stream = torch.cuda.current_stream()
    if o is None:
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.L), dtype=torch.float32, device=q.device)
    for _ in range(warmup):
        fa.forward(q, k, v, scale=w.scale, causal=w.causal, out=o, lse=lse, stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for s, e in ev:
        flush_buf.fill_(1)
        s.record(stream)
        fa.forward(q, k, v, scale=w.scale, causal=w.causal, out=o, lse=lse, stream=stream)
        e.record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in ev]


def time_splitkv(fa, torch, q, k, v, w, n_splits, steps, warmup, flush_buf):
    """Per-step device time (ms) of ``fa.forward_splitkv`` (split pass + merge)."""
    stream = torch.cuda.current_stream()
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.L), dtype=torch.float32, device=q.device)
    ws = torch.empty(fa.fa_splitkv_workspace_bytes(w.B, w.H, w.L, w.d, n_splits),
                     dtype=torch.uint8, device=q.device)
    run = lambda: fa.forward_splitkv(q, k, v, n_splits, scale=w.scale, causal=w.causal, out=o,
                                     lse=lse, workspace=ws, stream=stream)
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for s_, e_ in ev:
        flush_buf.fill_(1)
        s_.record(stream)
        run()
        e_.record(stream)
    torch.cuda.synchronize()
    return [s_.elapsed_time(e_) for s_, e_ in ev]


def time_backward(fa, torch, w, dev, steps, warmup, flush_buf):
    """Per-step device time (ms) of ``fa.backward`` (row pre-pass, gradient
    kernel, dQ conversion) on device-generated seeded inputs; O and LSE come
    from the forward, dO is a seeded normal.  L2 flushed before each step."""
    q, k, v = device_inputs(w, dev, torch)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed + 1000)
    do = torch.randn(q.shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    stream = torch.cuda.current_stream()
    o, lse = fa.forward(q, k, v, scale=w.scale, causal=w.causal, stream=stream)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.L, w.d), dtype=torch.uint8,
                     device=dev)
    run = lambda: fa.backward(q, k, v, o, lse, do, scale=w.scale, causal=w.causal, dq=dq, dk=dk,
                              dv=dv, workspace=ws, stream=stream)
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for s_, e_ in ev:
        flush_buf.fill_(1)
        s_.record(stream)
        run()
        e_.record(stream)
    torch.cuda.synchronize()
    return [s_.elapsed_time(e_) for s_, e_ in ev]


def time_fp8(fa, torch, w, dev, steps, warmup, flush_buf):
    """Per-step device time (ms) of the FP8 forward (``fa.forward_fp8`` on
    pre-quantised Q and K) and of the quantisation of Q and K; L2 flushed
    before each step."""
    q, k, v = device_inputs(w, dev, torch)
    stream = torch.cuda.current_stream()
    q8, qs = fa.quantize_fp8(q, stream=stream)
    k8, ks = fa.quantize_fp8(k, stream=stream)
    o = torch.empty_like(v)
    lse = torch.empty((w.B, w.H, w.L), dtype=torch.float32, device=dev)
    fwd = lambda: fa.forward_fp8(q8, k8, v, qs, ks, scale=w.scale, causal=w.causal, out=o, lse=lse,
                                 stream=stream)
    quant = lambda: (fa.quantize_fp8(q, codes=q8, scales=qs, stream=stream),
                     fa.quantize_fp8(k, codes=k8, scales=ks, stream=stream))
    out = []
    for run in (fwd, quant):
        for _ in range(warmup):
            run()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for s_, e_ in ev:
            flush_buf.fill_(1)
            s_.record(stream)
            run()
            e_.record(stream)
        torch.cuda.synchronize()
        out.append([s_.elapsed_time(e_) for s_, e_ in ev])
    return out


def backward_line(fa, w, t, peaks):
    mean = sum(t) / len(t)
    f = fa.flops_bwd(w.B, w.H, w.L, w.d, w.causal)
    tf = f / (mean * 1e-3) / 1e12
    traffic, src = read_traffic(w.name, "bwd")
    return {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "d": w.d, "causal": w.causal,
            "ms_mean": round(mean, 4), "ms_min": round(min(t), 4), "tflops": round(tf, 1),
            "frac_of_peak": round(tf / peaks["bf16_tflops"], 4), "steps": len(t),
            "gradient_kernel_dram_bytes": traffic, "traffic_source": src}


def splits_for(fa, w, sms):
    """The library's recommended split count (``fa_splitkv_splits``): as
    many splits as keep the CTAs within one wave (two when causal)."""
    return fa.fa_splitkv_splits(w.B, w.H, w.L, w.d, w.causal, sms)


# Shapes whose single-pass grid underfills the GPU (one head, long rows):
# where the split-KV path is meant to help.
SPLITKV_SHAPES = [
    ("B1_H1_L8192_d128", 1, 1, 8192, 128, False),
    ("B1_H1_L16384_d64", 1, 1, 16384, 64, False),
    ("B1_H1_L32768_d128_causal", 1, 1, 32768, 128, True),
]


def time_e2e(fa, torch, host, w, steps, warmup, flush_buf, dev):
    """End-to-end per-step time (ms) through the public host-buffer call
    ``fa.forward_host`` (the C-ABI ``fa_fwd_host``): every step copies its
    Q, K, V (pinned, back to back: one copy) to the device, runs the forward
    and copies O and LSE (back to back: one copy) to pinned host memory.

    Steps alternate between two device workspaces on two streams, as a
    caller streaming batches would, so the copies of one step overlap the
    kernel and copies of the previous one (the host link is full-duplex).
    Returns (pipelined per-step times over the K steps, serial per-step
    times with an L2 flush before each, h2d bytes, d2h bytes)."""
    shape = (w.B, w.H, w.L, w.d)
    nb = w.n_elem * 2                      # bytes of one bf16 tensor
    lb = w.B * w.H * w.L * 4               # bytes of LSE
    h_in = torch.empty(3 * nb, dtype=torch.uint8).pin_memory()
    for i, x in enumerate(host):
        h_in[i * nb:(i + 1) * nb].copy_(x.reshape(-1).view(torch.uint8))
    qh, kh, vh = (h_in[i * nb:(i + 1) * nb].view(torch.bfloat16).view(shape) for i in range(3))
    h_out = [torch.empty(nb + lb, dtype=torch.uint8).pin_memory() for _ in range(2)]
    outs = [(ho[:nb].view(torch.bfloat16).view(shape),
             ho[nb:].view(torch.float32).view(w.B, w.H, w.L)) for ho in h_out]
    need = fa.fa_fwd_host_workspace_bytes(w.B, w.H, w.L, w.d)
    ws = [torch.empty(need, dtype=torch.uint8, device=dev) for _ in range(2)]
    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    main = torch.cuda.current_stream()

    def step(i, stream):
        o, l = outs[i % 2]
        fa.forward_host(qh, kh, vh, scale=w.scale, causal=w.causal, out=o, lse=l,
                        workspace=ws[i % 2], stream=stream, device=dev)

    def pipelined(k):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(main)
        for st in streams:
            st.wait_stream(main)
        for i in range(k):
            step(i, streams[i % 2])
        for st in streams:
            main.wait_stream(st)
        end.record(main)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    pipelined(max(3, warmup))
    total = pipelined(steps)
    pipe = [total / steps] * steps
    # serial reference: one step at a time, L2 flushed before each
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i, (s_, e_) in enumerate(ev):
        flush_buf.fill_(1)
        s_.record(main)
        step(i, main)
        e_.record(main)
    torch.cuda.synchronize()
    serial = [s_.elapsed_time(e_) for s_, e_ in ev]
    return pipe, serial, 3 * nb, nb + lb


def max_over_ranks(values, world, dist=None, device=None):
    """Element-wise max of per-rank timing totals across the process group
    (the slowest rank sets the job's time); identity for one rank."""
    if world <= 1:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_tflops(world, flops_per_step, steps, total_ms):
    """TFLOP/s of the whole job: every rank runs ``steps`` steps of its own
    replica, and the job takes the slowest rank's time."""
    return world * flops_per_step * steps / (total_ms * 1e-3) / 1e12


def forward_line(w, t, peaks):
    """Compact per-workload forward entry (kept short: the line's tail)."""
    st = step_stats(t)
    tf = w.flops / (st["ms_mean"] * 1e-3) / 1e12
    return {"workload": w.name, "ms_mean": st["ms_mean"], "ms_median": st["ms_median"],
            "tflops": round(tf, 1), "frac_of_peak": round(tf / peaks["bf16_tflops"], 4),
            "steps": len(t)}


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import exact_tiled_attention_09_gb300 as fa
    from fa_inputs import WORKLOADS, make_qkv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.library()
    peaks, peak_src = read_peaks()

    w = WORKLOADS[args.workload]
    if args.device_inputs:
        q, k, v = device_inputs(w, dev, torch)
        host = tuple(x.cpu().pin_memory() for x in (q, k, v))
    else:
        qb, kb, vb = make_qkv(w)
        as_t = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)
        host = tuple(as_t(x).pin_memory() for x in (qb, kb, vb))
        q, k, v = (x.to(dev) for x in host)
    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    extras = []
    splitkv = []
    backward = []
    fp8 = []
    fp8_peak = FP8_OVER_BF16 * peaks["bf16_tflops"]
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        ms = time_forward(fa, torch, q, k, v, w, args.steps, args.warmup, flush_buf)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e2e_ms, e2e_serial, h2d, d2h = time_e2e(fa, torch, host, w, args.steps, args.warmup,
                                                 flush_buf, dev)
        if rank == 0 and not args.no_extra:
            for name, wx in WORKLOADS.items():
                if name == w.name:
                    extras.append(forward_line(wx, ms, peaks))
                    continue
                qx, kx, vx = device_inputs(wx, dev, torch)
                steps = max(3, min(args.extra_steps, int(2e13 / wx.flops)))
                t = time_forward(fa, torch, qx, kx, vx, wx, steps, 3, flush_buf)
                extras.append(forward_line(wx, t, peaks))
                del qx, kx, vx
            for name, wx in WORKLOADS.items():
                steps = max(3, min(args.extra_steps, int(2e13 / wx.flops)))
                tf8, tq = time_fp8(fa, torch, wx, dev, steps, 3, flush_buf)
                m8, mq = sum(tf8) / len(tf8), sum(tq) / len(tq)
                tr8, tr8_src = read_traffic(name, "fwd_fp8")
                t8 = wx.flops / (m8 * 1e-3) / 1e12
                fp8.append({"workload": name, "ms_mean": round(m8, 4),
                            "ms_min": round(min(tf8), 4),
                            "attention_kernel_dram_bytes": tr8, "traffic_source": tr8_src,
                            "tflops": round(t8, 1),
                            "frac_of_fp8_peak": round(t8 / fp8_peak, 4),
                            "frac_of_bf16_peak": round(t8 / peaks["bf16_tflops"], 4),
                            "quantize_qk_ms": round(mq, 4), "steps": steps})
            for name, wx in WORKLOADS.items():
                steps = max(3, min(args.extra_steps,
                                   int(5e13 / fa.flops_bwd(wx.B, wx.H, wx.L, wx.d, wx.causal))))
                t = time_backward(fa, torch, wx, dev, steps, 3, flush_buf)
                backward.append(backward_line(fa, wx, t, peaks))
            from fa_inputs import AttentionWorkload
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            for name, B, H, L, d, causal in SPLITKV_SHAPES:
                wx = AttentionWorkload(name, B, H, L, d, causal, 1.0 / math.sqrt(d), 100 + L)
                qx, kx, vx = device_inputs(wx, dev, torch)
                S = splits_for(fa, wx, sms)
                steps = max(3, min(args.extra_steps, int(2e13 / wx.flops)))
                t1 = time_forward(fa, torch, qx, kx, vx, wx, steps, 3, flush_buf)
                t2 = time_splitkv(fa, torch, qx, kx, vx, wx, S, steps, 3, flush_buf)
                m1, m2 = sum(t1) / len(t1), sum(t2) / len(t2)
                splitkv.append({"workload": name, "B": B, "H": H, "L": L, "d": d,
                                "causal": causal, "n_splits": S,
                                "single_pass_ms": round(m1, 4), "splitkv_ms": round(m2, 4),
                                "single_pass_tflops": round(wx.flops / (m1 * 1e-3) / 1e12, 1),
                                "splitkv_tflops": round(wx.flops / (m2 * 1e-3) / 1e12, 1),
                                "steps": steps})
                del qx, kx, vx
    if fa.fa_device_status(None, clear=True) != fa.FA_OK:
        raise RuntimeError("a kernel wait timed out during the benchmark")

    # CPU baseline after the GPU timing (rank 0 only), so the timed region
    # does not start on a GPU that sat idle for the seconds it takes
    cpu = None
    if rank == 0 and not args.no_cpu_baseline and not args.device_inputs:
        cpu = cpu_baseline(w, qb, kb, vb)

    total_ms, total_e2e = max_over_ranks([sum(ms), sum(e2e_ms)], world, dist, dev)
    flops_step = w.flops
    value = whole_job_tflops(world, flops_step, args.steps, total_ms)
    e2e_value = whole_job_tflops(world, flops_step, args.steps, total_e2e)
    st = step_stats(ms)
    achieved = flops_step / (st["ms_mean"] * 1e-3) / 1e12
    traffic, traffic_src = read_traffic(w.name)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded SplitMix64 + Box-Muller normals rounded to bf16)",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "d": w.d,
                       "causal": w.causal, "scale": w.scale,
                       "l2": "flushed before every timed step (512 MiB device write, untimed)",
                       "parallelism": f"replicas x{world} (no exchange step)"},
            "percent_of_peak": round(100 * value / world / peaks["bf16_tflops"], 2),
            "nominal_peak": {"value": NOMINAL_BF16_TFLOPS, "unit": "TFLOP/s",
                             "source": "NVIDIA nominal dense bf16 per GB300 (2:4-sparse figure "
                                       "halved); second denominator, not the roofline's",
                             "frac": round(achieved / NOMINAL_BF16_TFLOPS, 4)},
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(achieved / peaks["bf16_tflops"], 4),
                         "peak_source": f"{peak_src} bf16_tflops (burst; kernel timed alone)",
                         "traffic": traffic, "traffic_source": traffic_src,
                         "algorithmic_bytes": w.algorithmic_bytes,
                         "kernel": f"fa_fwd_kernel<{w.d},{str(w.causal).lower()}>", **st},
            "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(total_e2e / args.steps, 5),
                    "api": "fa_fwd_host (C ABI, pinned host buffers)",
                    "pipelining": "steps alternate two workspaces on two streams; each "
                                  "step's H2D, kernel and D2H are in the timed region",
                    "serial_ms_per_step": round(sum(e2e_serial) / len(e2e_serial), 5),
                    "serial_value": round(world * flops_step * len(e2e_serial)
                                          / (sum(e2e_serial) * 1e-3) / 1e12, 3),
                    "l2": "inputs are re-copied from the host every step (no flush "
                          "in the pipelined run; the serial run flushes); a copy larger "
                          "than L2 leaves its last part L2-resident for the kernel that "
                          "follows, which is why the pipelined step can beat the "
                          "flushed kernel-only step"},
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
            "fp8_peak": {"value": fp8_peak, "unit": "TFLOP/s",
                         "source": f"{peak_src} bf16_tflops x {FP8_OVER_BF16} (nominal dense "
                                   "fp8/bf16 rate ratio)"},
            "splitkv": splitkv,
            "fp8": fp8,
            "backward": backward,
            # last: the bf16 forward on every configuration (compact entries)
            "workloads": extras,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_profile_bwd(args):
    """Time only the backward pass of one workload (for profiler captures)."""
    import torch

    import exact_tiled_attention_09_gb300 as fa
    from fa_inputs import WORKLOADS

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fa.library()
    peaks, _ = read_peaks()
    w = WORKLOADS[args.profile_bwd]
    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    t = time_backward(fa, torch, w, dev, args.steps, args.warmup, flush_buf)
    if fa.fa_device_status(None, clear=True) != fa.FA_OK:
        raise RuntimeError("a kernel wait timed out during the benchmark")
    print(json.dumps({"backward": backward_line(fa, w, t, peaks)}), flush=True)


def run_profile_fp8(args):
    """Time only the FP8 forward of one workload (for profiler captures)."""
    import torch

    import exact_tiled_attention_09_gb300 as fa
    from fa_inputs import WORKLOADS

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fa.library()
    w = WORKLOADS[args.profile_fp8]
    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    t8, tq = time_fp8(fa, torch, w, dev, args.steps, args.warmup, flush_buf)
    if fa.fa_device_status(None, clear=True) != fa.FA_OK:
        raise RuntimeError("a kernel wait timed out during the benchmark")
    m8 = sum(t8) / len(t8)
    print(json.dumps({"fp8": {"workload": w.name, "ms_mean": round(m8, 4),
                              "tflops": round(w.flops / (m8 * 1e-3) / 1e12, 1),
                              "quantize_qk_ms": round(sum(tq) / len(tq), 4)}}), flush=True)


def run_reference(args):
    """The fp64 oracle on the host cores, same metric/config (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    from fa_inputs import WORKLOADS, make_qkv

    w = WORKLOADS[args.workload]
    qb, kb, vb = make_qkv(w)
    BH = w.B * w.H
    # bounded sample per step: about one second of host work
    heads, rows = sample_size(w, qb, kb, vb, 1.0)
    for _ in range(args.warmup):
        oracle_sample_run(w, qb, kb, vb, heads, rows)
    total_t, total_f = 0.0, 0.0
    for _ in range(args.steps):
        t, f = oracle_sample_run(w, qb, kb, vb, heads, rows)
        total_t += t
        total_f += f
    value = total_f / total_t / 1e12
    cores = os.cpu_count() or 1
    what = (f"query rows 0..{rows - 1} of head 0" if heads == 1 and rows < w.L
            else f"{heads} of {BH} whole heads")
    line = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total_t / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64 + Box-Muller normals rounded to bf16)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "d": w.d,
                   "causal": w.causal, "scale": w.scale},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{what} of {w.name} per step (every key), fp64"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--extra-steps", type=int, default=30)
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--device-inputs", action="store_true",
                    help="draw the headline inputs with a seeded device generator "
                         "(no CPU baseline then); used for profiling large workloads")
    ap.add_argument("--profile-bwd", metavar="WORKLOAD", default=None,
                    help="time only the backward pass of WORKLOAD and print its line "
                         "(for profiler captures; not the benchmark line)")
    ap.add_argument("--profile-fp8", metavar="WORKLOAD", default=None,
                    help="time only the FP8 forward of WORKLOAD (for profiler captures)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.profile_bwd:
        run_profile_bwd(args)
    elif args.profile_fp8:
        run_profile_fp8(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
