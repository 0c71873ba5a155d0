#!/usr/bin/env python3
"""Benchmark of the gated delta rule hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload prefill|long|million|decode|varlen] [--no-cpu-baseline]

One JSON line on rank 0.  A "step" of the default workload is one chunked
prefill over B=4, H=16, T=4096, d=128, bf16 (cumulative decay, WY/UT
transform, state pass and output); ``value`` is prefill tokens/s (B*T per
step).  The same line carries a ``decode`` object for the single-token decode
workload (N=256 sequences x H=32 heads, one token per step), because the
metric asks for both, a ``backward`` object (the gradients of the prefill
workload), and ``long`` (B=1, H=32, T=65536) and ``million`` (B=1, H=16,
T=1,048,576) objects for the two long prefill workloads, each with its own
roofline and oracle baseline, and ``mla``: one decode step of gated multi-head
latent attention (N=32 sequences, H=64 heads, 32768 cached latents of 512 values).  ``--workload varlen`` times the packed variable-length
prefill instead: 32 sequences of seeded lengths in [16, 4096] (34,599 tokens),
H=16, through ``chunk_fwd_varlen``; ``value`` is packed tokens/s.

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events on
the launching stream with an L2 flush (a 256 MB write) between steps, outside
the events.  Ranks are independent replicas (weak scaling): a barrier and a
device synchronise bracket the timed region, and the slowest rank's time
counts.  ``e2e`` repeats the measurement with the inputs in pinned host memory
copied in, and the result copied out, inside the timed region.

``--impl reference`` times the fp64 CPU oracle (the only reference this
project has) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gated_delta_rule_gdr_gb300 import inputs as I  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def prefill_algorithmic(w: I.Workload):
    """Algorithmic bytes and chunked FLOPs of one prefill call.

    Bytes: q, k, v and out once each, g and beta once, the fp32 state read once
    (if given) and written once.  FLOPs: per token-head, 6 dk dv for the three
    state products plus 2 C (3 dk + 2 dv) for the five C x C tile products,
    counted as full dense tiles as the chunked method computes them."""
    es = 2 if w.dtype == "bf16" else 4
    n_th = w.B * w.H * w.T
    by = n_th * ((2 * w.dk + 2 * w.dv) * es + 8)
    by += w.B * w.H * w.dk * w.dv * 4 * ((1 if w.init_std is not None else 0) + 1)
    fl = n_th * (6 * w.dk * w.dv + 2 * w.chunk * (3 * w.dk + 2 * w.dv))
    return by, fl


def varlen_algorithmic(w: I.Workload, lengths):
    """Bytes and FLOPs of one packed call: the prefill counts over total_T tokens,
    with one fp32 state read and written per (sequence, head)."""
    es = 2 if w.dtype == "bf16" else 4
    n_th = sum(lengths) * w.H
    by = n_th * ((2 * w.dk + 2 * w.dv) * es + 8)
    by += len(lengths) * w.H * w.dk * w.dv * 4 * ((1 if w.init_std is not None else 0) + 1)
    fl = n_th * (6 * w.dk * w.dv + 2 * w.chunk * (3 * w.dk + 2 * w.dv))
    return by, fl


def decode_algorithmic(w: I.Workload):
    """Bytes of one decode step: state read + written (fp32), q, k, v, out, g, beta."""
    es = 2 if w.dtype == "bf16" else 4
    per = 2 * w.dk * w.dv * 4 + (2 * w.dk + 2 * w.dv) * es + 8
    return w.B * w.H * per


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"), parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def committed_traffic(kernel: str, source_files, workload: str | None = None):
    """ncu DRAM bytes per launch committed under profiles/ (keyed "kernel @ workload",
    or by the kernel alone), valid only while the kernel's source is unchanged (sha256
    of its files)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(f"{kernel} @ {workload}") if workload else None
    ent = ent or d.get(kernel)
    if not ent:
        return None
    h = hashlib.sha256()
    for fn in source_files:
        with open(os.path.join(ROOT, fn), "rb") as f:
            h.update(f.read())
    if ent.get("source_sha256") != h.hexdigest():
        return None
    return ent.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- our arm
def time_steps(fn, K, W, flush, stream, prime=True):
    """Run W warm-ups then K timed steps; per-step CUDA-event times in ms.

    prime: queue a ~1 ms device spin ahead of the timed steps, so that the first
    step's start event is not recorded on an idle device while the host is still
    enqueueing that step (after the synchronize, the host's launch overhead would
    otherwise land inside the first step's device time).  The end-to-end legs run
    unprimed."""
    for _ in range(W):
        if flush is not None:   # the timed steps' flush kernel is warm too
            flush.zero_()
        fn(-1)
    torch.cuda.synchronize()
    if prime:
        with torch.cuda.stream(stream):
            if hasattr(torch.cuda, "_sleep"):
                torch.cuda._sleep(2_000_000)
            else:   # ~1 ms of device work by other means
                a = torch.ones((4096, 4096), device=stream.device, dtype=torch.bfloat16)
                for _ in range(8):
                    a = a @ a * (1.0 / 4096)
    times = []
    for i in range(K):
        if flush is not None:
            flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn(i)
        e.record(stream)
        times.append((s, e))
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in times]


def time_two_streams(fn, K, W, dev):
    """K steps fn(i, stream) alternating over two streams, after W warm-ups; the
    device time from an event before the first step to one after both streams have
    drained, per step (a list of K equal values)."""
    sts = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
    for i in range(W):
        fn(i, sts[i % 2])
    torch.cuda.synchronize()
    start, mid, end = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    start.record(sts[0])
    sts[1].wait_event(start)
    for i in range(K):
        fn(i, sts[i % 2])
    mid.record(sts[1])
    sts[0].wait_event(mid)
    end.record(sts[0])
    torch.cuda.synchronize()
    return [start.elapsed_time(end) / K] * K


def bench_prefill(gdr, w, K, W, dev, flush, stream, workspace="auto"):
    x = I.prefill_inputs(w, device=dev)
    out = torch.empty((w.B, w.H, w.T, w.dv), dtype=w.torch_dtype(), device=dev)
    fin = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)

    # the workspace of the two-kernel path, held across steps like the inputs
    nws = gdr.chunk_fwd_workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.chunk, w.torch_dtype())
    ws = torch.empty(nws, dtype=torch.uint8, device=dev) if (workspace and nws) else None

    def step(_):
        gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, x["init_state"],
                      chunk=w.chunk, out=out, final_state=fin, workspace=ws)

    ms = time_steps(step, K, W, flush, stream)

    # end to end: pinned host inputs in, output and final state out, every step, through
    # the host-buffer entry point; two streams with a device buffer each, so one step's
    # copies overlap the other's kernels
    host = {n: (None if t is None else t.cpu().pin_memory()) for n, t in x.items()}
    del x, out, fin, ws
    nbuf = gdr.chunk_fwd_host_buffer_size(w.B, w.H, w.T, w.dk, w.dv, w.chunk, w.torch_dtype())
    bufs = [torch.empty(nbuf, dtype=torch.uint8, device=dev) for _ in range(2)]
    houts = [torch.empty((w.B, w.H, w.T, w.dv), dtype=w.torch_dtype(), pin_memory=True)
             for _ in range(2)]
    hfins = [torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, pin_memory=True)
             for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = houts[0].numel() * houts[0].element_size() + hfins[0].numel() * hfins[0].element_size()

    def e2e_step(i, st):
        gdr.chunk_fwd_host(host["q"], host["k"], host["v"], host["g"], host["beta"], w.a_min,
                           host["init_state"], houts[i % 2], hfins[i % 2], bufs[i % 2],
                           chunk=w.chunk, stream=st)

    ms_e2e = time_two_streams(e2e_step, max(3, K // 2), 2, dev)
    return ms, ms_e2e, h2d, d2h


def bench_varlen(gdr, w, K, W, dev, flush, stream, workspace="auto"):
    lengths = I.varlen_lengths(w)
    x = I.varlen_inputs(w, lengths, device=dev)
    del x["seqs"]
    total_T, S = sum(lengths), len(lengths)
    out = torch.empty((total_T, w.H, w.dv), dtype=w.torch_dtype(), device=dev)
    fin = torch.empty((S, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)

    nws = gdr.chunk_fwd_varlen_workspace_size(S, w.H, total_T, w.dk, w.dv, w.chunk, w.torch_dtype())
    ws = torch.empty(nws, dtype=torch.uint8, device=dev) if (workspace and nws) else None

    def step(_):
        gdr.chunk_fwd_varlen(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min,
                             x["cu_seqlens"], x["init_state"], chunk=w.chunk, out=out,
                             final_state=fin, workspace=ws)

    ms = time_steps(step, K, W, flush, stream)

    # end to end: every packed input (cu_seqlens included) in, output and final states out
    host = {n: (None if t is None else t.cpu().pin_memory()) for n, t in x.items()}
    dx = {n: (None if t is None else torch.empty_like(t)) for n, t in x.items()}
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    hfin = torch.empty(fin.shape, dtype=fin.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = hout.numel() * hout.element_size() + hfin.numel() * hfin.element_size()

    def e2e_step(_):
        for n, t in host.items():
            if t is not None:
                dx[n].copy_(t, non_blocking=True)
        gdr.chunk_fwd_varlen(dx["q"], dx["k"], dx["v"], dx["g"], dx["beta"], w.a_min,
                             dx["cu_seqlens"], dx["init_state"], chunk=w.chunk, out=out,
                             final_state=fin, workspace=ws)
        hout.copy_(out, non_blocking=True)
        hfin.copy_(fin, non_blocking=True)

    ms_e2e = time_steps(e2e_step, max(3, K // 2), 2, flush, stream, prime=False)
    return ms, ms_e2e, h2d, d2h


def bench_prefill_leg(gdr, w, K, W, dev, stream):
    """Device-resident prefill of a long workload through the binding's default path
    (the caller-owned workspace of the two-kernel path); per-step CUDA-event times.
    Its inputs (2.2 GB, 17.3 GB) are far larger than L2, so no flush is needed."""
    x = I.prefill_inputs(w, device=dev)
    out = torch.empty((w.B, w.H, w.T, w.dv), dtype=w.torch_dtype(), device=dev)
    fin = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
    nws = gdr.chunk_fwd_workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.chunk, w.torch_dtype())
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)

    def step(_):
        gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, x["init_state"],
                      chunk=w.chunk, out=out, final_state=fin, workspace=ws)

    ms = time_steps(step, K, W, None, stream)
    return ms, x


def prefill_leg_line(gdr, w, ms, pk, pk_kind, world, max_over_ranks):
    """The JSON object of a prefill leg: value, roofline of its kernels, launches."""
    path = gdr.chunk_fwd_path(w.B, w.H, w.T, w.dk, w.dv, w.chunk, w.a_min, w.torch_dtype())
    kname, srcs, nk = path_kernels(path)
    mean = statistics.mean(ms)
    by, fl = prefill_algorithmic(w)
    gbs = by / (mean * 1e-3) / 1e9
    return {
        "metric": "prefill tokens/s", "workload": w.name,
        "value": round(world * w.B * w.T / (max_over_ranks(mean) * 1e-3), 1), "unit": "tokens/s",
        "ms_per_step": round(mean, 4), "steps": len(ms), "path": gdr.PATHS.get(path, str(path)),
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": round(gbs, 1),
                     "peak": pk["hbm_gbs"], "peak_kind": pk_kind, "unit": "GB/s",
                     "frac": round(gbs / pk["hbm_gbs"], 4),
                     "traffic": committed_traffic(kname, srcs, w.name),
                     "algorithmic_bytes": by, "algorithmic_flops": fl,
                     "achieved_tflops": round(fl / (mean * 1e-3) / 1e12, 2),
                     "nominal_hbm_frac": round(gbs / 7900.0, 4)},
        "l2": "inputs far larger than L2, no flush",
        "gpu_launches": nk * len(ms),
        "ms_per_step_all": [round(t, 4) for t in ms],
    }


CSRC = "gated_delta_rule_gdr_gb300/csrc/"
# the four launches of one backward step on the bf16, d = 128, chunk 64 shape: the training
# forward's kernels into the workspace (its chain, without output products, keeps the states
# and W tiles), then the saved-state backward
BWD_KERNELS = ("backward: chunk_prep_kernel<true> + chain_kernel<64> (states only) + bwd_passes_vc_kernel + "
               "bwd_chunk_tc_kernel")
# one training step: the forward with saves (two-kernel path) and the saved-state backward
# (the forward's prep kernel also writes T, P and the row scalars, so the backward runs
# neither the decay nor the tiles kernel)
TRAIN_KERNELS = ("training: chunk_prep_kernel<true> + chain_kernel<64> + bwd_passes_vc_kernel + "
                 "bwd_chunk_tc_kernel")
BWD_SRCS = [CSRC + "gdr_bwd.cu", CSRC + "gdr_bwd_tc.cu", CSRC + "gdr_staged.cu"]
_COMMON = [CSRC + "gdr_fused_common.cuh", CSRC + "gdr_sm100.cuh"]


def path_kernels(path):
    """(kernel name as ncu lists it, source files, launches per call) of a prefill path."""
    return {
        1: ("staged: decay_kernel + wy_kernel + state_kernel + output_kernel",
            [CSRC + "gdr_staged.cu"], 4),
        2: ("fused_prefill_kernel", [CSRC + "gdr_fused.cu"] + _COMMON, 1),
        3: ("fused_pair_kernel", [CSRC + "gdr_fused_pair.cu"] + _COMMON, 1),
        # the two-kernel step is timed as one unit (its two launches back to back)
        4: ("chunk_prep_kernel + chain_kernel<64>",
            [CSRC + "gdr_prep.cu", CSRC + "gdr_chain.cu"] + _COMMON, 2),
        5: ("chunk_prep_kernel + chain_kernel<128>",
            [CSRC + "gdr_prep.cu", CSRC + "gdr_chain.cu"] + _COMMON, 2),
        6: ("onepass_kernel", [CSRC + "gdr_onepass.cu"], 1),
        # sequence segments: preparation, the segment maps, the scan, every segment's chain
        7: ("chunk_prep_kernel + seg_pass1_kernel + seg_scan_kernel + chain_kernel",
            [CSRC + "gdr_prep.cu", CSRC + "gdr_segment.cu", CSRC + "gdr_chain.cu"] + _COMMON, 4),
    }[path]


def mla_algorithmic(w: I.MlaWorkload):
    """Bytes and FLOPs of one latent-attention decode step: the latent cache, the
    queries, W_uv, the gate and the output once each; QK and PV over every cached
    token (2 dc MACs each per head) plus the up-projection."""
    by = (w.N * w.L * w.dc * 2 + w.N * w.H * w.dc * 2 + w.H * w.dh * w.dc * 2
          + w.N * w.H * w.dh * (4 + 2))
    fl = 4 * w.N * w.H * w.L * w.dc + 2 * w.N * w.H * w.dh * w.dc
    return by, fl


def bench_mla(gdr, w, K, W, dev, stream):
    """One decode step of gated latent attention over the device-resident cache (1 GiB,
    far larger than L2: no flush)."""
    x = I.mla_inputs(w, device=dev)
    ws = torch.empty(max(gdr.mla_decode_workspace_size(w.N, w.H, w.L, w.dc, w.dh), 16),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((w.N, w.H, w.dh), dtype=torch.bfloat16, device=dev)

    def step(_):
        gdr.mla_decode(x["q_abs"], x["ckv"], x["seqlens"], x["w_uv"], x["gate"], w.scale, out=out,
                       workspace=ws)

    return time_steps(step, K, W, None, stream), x


def cpu_baseline_mla(w, x, budget_s=6.0):
    """The fp64 oracle on whole sequences of the decode step, every head, until about
    budget_s of work; value in the leg's unit (sequences' tokens per second)."""
    import oracle
    cores = os.cpu_count() or 1
    n, dt = 0, 0.0
    while dt < budget_s and n < w.N:
        sub = {k: (t if k == "w_uv" else t[n:n + 1]).cpu() for k, t in x.items()}
        t0 = time.perf_counter()
        oracle.mla_decode(sub["q_abs"], sub["ckv"], sub["seqlens"], sub["w_uv"], sub["gate"],
                          w.scale, nthreads=cores)
        dt += time.perf_counter() - t0
        n += 1
    return {"value": n / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} of {w.N} sequences, all {w.H} heads, {w.L} cached tokens each "
                      f"({dt:.2f} s); value = decoded tokens per second"}


def bench_decode(gdr, w, K, W, dev, flush, stream):
    state = I.decode_state(w, device=dev)
    nsteps = max(K, 1)
    xs = [I.decode_step_inputs(w, s % w.steps, device=dev) for s in range(min(nsteps, w.steps))]
    out = torch.empty((w.B, w.H, w.dv), dtype=w.torch_dtype(), device=dev)

    def step(i):
        x = xs[i % len(xs)]
        gdr.decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, state, out=out)

    # the state (537 MB) is larger than L2: no flush needed between decode steps
    ms = time_steps(step, K, W, None, stream)

    hx = [{n: t.cpu().pin_memory() for n, t in x.items()} for x in xs[:4]]
    dx = {n: torch.empty_like(t) for n, t in xs[0].items()}
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in hx[0].values())
    d2h = hout.numel() * hout.element_size()

    def e2e_step(i):
        for n, t in hx[i % len(hx)].items():
            dx[n].copy_(t, non_blocking=True)
        gdr.decode_step(dx["q"], dx["k"], dx["v"], dx["g"], dx["beta"], w.a_min, state, out=out)
        hout.copy_(out, non_blocking=True)

    ms_e2e = time_steps(e2e_step, K, 2, None, stream, prime=False)
    return ms, ms_e2e, h2d, d2h


def backward_algorithmic(w: I.Workload):
    """Bytes one backward step must move at the least: q, k, v, g, beta and d_out in,
    dq, dk, dv, dg, dbeta out per token and head; the initial state and d_final in and
    the initial state's gradient out per head."""
    es = 2 if w.dtype == "bf16" else 4
    per_tok = (2 * w.dk + w.dv) * es + w.dv * es + (2 * w.dk + w.dv) * es + 4 * 4
    return w.B * w.H * (w.T * per_tok + 3 * w.dk * w.dv * 4)


def bench_backward(gdr, w, K, W, dev, flush, stream):
    x = I.prefill_inputs(w, device=dev)
    ct = I.cotangents(w, device=dev)
    nws = gdr.chunk_bwd_workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.chunk, w.torch_dtype())
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)

    def step(_):
        gdr.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, x["init_state"],
                      ct["d_out"], ct["d_final"], chunk=w.chunk, workspace=ws)

    return time_steps(step, K, W, flush, stream), nws


def bench_training(gdr, w, K, W, dev, flush, stream):
    """One training step of the prefill workload: the forward that saves its chunk states
    (gdr_chunk_fwd_train) and the backward that reads them (gdr_chunk_bwd_saved); each
    half is also timed alone."""
    x = I.prefill_inputs(w, device=dev)
    ct = I.cotangents(w, device=dev)
    td = w.torch_dtype()
    wsf = torch.empty(max(gdr.chunk_fwd_workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.chunk, td), 16),
                      dtype=torch.uint8, device=dev)
    wsb = torch.empty(max(gdr.chunk_bwd_workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.chunk, td), 16),
                      dtype=torch.uint8, device=dev)
    nsv = gdr.chunk_saved_size(w.B, w.H, w.T, w.dk, w.dv, w.chunk, td)
    saved = torch.empty(max(nsv, 16), dtype=torch.uint8, device=dev)
    out = torch.empty((w.B, w.H, w.T, w.dv), dtype=td, device=dev)
    fin = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)

    def fwd(_):
        gdr.chunk_fwd_train(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, x["init_state"],
                            out=out, final_state=fin, workspace=wsf, saved=saved)

    def bwd(_):
        gdr.chunk_bwd_saved(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, x["init_state"],
                            ct["d_out"], saved, ct["d_final"], workspace=wsb)

    def step(i):
        fwd(i)
        bwd(i)

    ms = time_steps(step, K, W, flush, stream)
    ms_f = time_steps(fwd, K, W, flush, stream)
    ms_b = time_steps(bwd, K, W, flush, stream)
    path = gdr.chunk_fwd_path(w.B, w.H, w.T, w.dk, w.dv, w.chunk, w.a_min, td, workspace=True)
    return ms, ms_f, ms_b, nsv, (4 if path == 7 else 2) + 2


def cpu_baseline_backward(w, budget_s=8.0):
    """The fp64 oracle's backward on a bounded sample of the prefill workload: all
    heads of sequence 0 over the first T_s tokens, T_s grown until ~budget_s."""
    import oracle
    x = I.prefill_inputs(w.with_(B=1), device="cpu")
    ct = I.cotangents(w.with_(B=1), device="cpu")
    cores = os.cpu_count() or 1
    Ts = 64
    while True:
        sub = {n: x[n][:, :, :Ts] for n in ("q", "k", "v", "g", "beta")}
        t0 = time.perf_counter()
        oracle.bwd(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], w.a_min,
                   x["init_state"], ct["d_out"][:, :, :Ts], ct["d_final"], nthreads=cores)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 4 or Ts >= w.T:
            break
        Ts = min(w.T, Ts * 4)
    return {"value": Ts / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"B=1 of {w.B}, all {w.H} heads, first {Ts} of {w.T} tokens "
                      f"({w.H * Ts} head-tokens in {dt:.2f} s); value = head-tokens/s / H"}


def cpu_baseline_prefill(w, budget_s=12.0, x=None):
    """fp64 oracle on a bounded sample of the prefill workload: all heads of
    sequence 0 over the first T_s tokens, T_s grown until ~budget_s of work.  x: the
    workload's inputs already drawn (on any device; the sample is sliced and copied)."""
    import oracle
    if x is None:
        x = I.prefill_inputs(w.with_(B=1), device="cpu")
    cores = os.cpu_count() or 1
    Ts = 128
    while True:
        sub = {n: x[n][:1, :, :Ts].cpu().contiguous() for n in ("q", "k", "v", "g", "beta")}
        init = None if x["init_state"] is None else x["init_state"][:1].cpu()
        t0 = time.perf_counter()
        oracle.fwd(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], w.a_min, init,
                   nthreads=cores)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 4 or Ts >= w.T:
            break
        Ts = min(w.T, Ts * 4)
    head_tok_s = w.H * Ts / dt
    return {"value": head_tok_s / w.H, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"B=1 of {w.B}, all {w.H} heads, first {Ts} of {w.T} tokens "
                      f"({w.H * Ts} head-tokens in {dt:.2f} s); value = head-tokens/s / H",
            "head_tokens_per_s": head_tok_s}


def oracle_varlen_sample(w, lengths, budget_s, cores):
    """The fp64 oracle over whole sequences of the packed workload, all heads, in
    the workload's order, until about budget_s of work; (tokens, seconds, count)."""
    import oracle
    tok, dt, n = 0, 0.0, 0
    for s, T in enumerate(lengths):
        x = I.prefill_inputs(w.with_(B=1, T=int(T), seed=w.seed * 1000 + s + 1), device="cpu")
        t0 = time.perf_counter()
        oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, x["init_state"],
                   nthreads=cores)
        dt += time.perf_counter() - t0
        tok += int(T)
        n += 1
        if dt >= budget_s:
            break
    return tok, dt, n


def cpu_baseline_varlen(w, budget_s=12.0):
    cores = os.cpu_count() or 1
    lengths = I.varlen_lengths(w)
    tok, dt, n = oracle_varlen_sample(w, lengths, budget_s, cores)
    return {"value": tok / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"the first {n} of {len(lengths)} sequences, all {w.H} heads "
                      f"({tok} of {sum(lengths)} tokens in {dt:.2f} s)"}


def cpu_baseline_decode(w, budget_s=8.0):
    import numpy as np
    import oracle
    cores = os.cpu_count() or 1
    state = I.decode_state(w, device="cpu").double().numpy().copy()
    steps, t_tot = 0, 0.0
    while t_tot < budget_s and steps < w.steps:
        x = I.decode_step_inputs(w, steps, device="cpu")
        t0 = time.perf_counter()
        oracle.decode(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, state, nthreads=cores)
        t_tot += time.perf_counter() - t0
        steps += 1
    return {"value": w.B * steps / t_tot, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{steps} of {w.steps} decode steps over all {w.B}x{w.H} (n,h)",
            "ms_per_step": 1e3 * t_tot / steps}


def rank_barrier(dist, sync=None):
    """The device's work done (sync), then every rank at the same point."""
    if sync is not None:
        sync()
    if dist is not None:
        dist.barrier()


def rank_max(dist, x: float) -> float:
    """The maximum of x over the ranks (x itself with one process): the timed region
    ends when the slowest replica ends."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_ours(args):
    import gated_delta_rule_gdr_gb300 as gdr
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    gdr.load(build_if_missing=True)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    pk, pk_kind = peaks()

    main_w = WORKLOAD_ARG[args.workload]
    prefill_family = main_w is I.PREFILL   # the backward and training legs follow its sizes
    varlen = main_w is I.VARLEN
    if main_w.steps == 0 and not varlen and (args.B or args.H or args.T):
        # a smaller case of the same prefill workload (for profiling); the line names it
        main_w = main_w.with_(B=args.B or main_w.B, H=args.H or main_w.H, T=args.T or main_w.T,
                              name=f"{main_w.name} (B={args.B or main_w.B} H={args.H or main_w.H} "
                                   f"T={args.T or main_w.T})")

    def barrier():
        rank_barrier(dist, torch.cuda.synchronize)

    def max_over_ranks(x):
        return rank_max(dist, x)

    result = {}
    with ClockSampler(dev.index) as clocks:
        barrier()
        t_wall0 = time.perf_counter()
        if varlen:
            ms, ms_e2e, h2d, d2h = bench_varlen(gdr, main_w, args.steps, args.warmup, dev, flush,
                                                stream, workspace=not args.single_launch)
        elif main_w.steps == 0:
            ms, ms_e2e, h2d, d2h = bench_prefill(gdr, main_w, args.steps, args.warmup, dev, flush,
                                                 stream, workspace=not args.single_launch)
        else:
            ms, ms_e2e, h2d, d2h = bench_decode(gdr, main_w, args.steps, args.warmup, dev, flush,
                                                stream)
        barrier()
        wall = time.perf_counter() - t_wall0
        dec = None
        if main_w.steps == 0 and not varlen and not args.no_decode:
            dec = bench_decode(gdr, I.DECODE, args.decode_steps, args.warmup, dev, flush, stream)
            barrier()
        bwd = None
        if prefill_family and not args.no_backward:
            bwd = bench_backward(gdr, main_w, max(3, args.steps // 2), 3, dev, flush, stream)
            barrier()
        train = None
        if prefill_family and not args.no_backward:
            train = bench_training(gdr, main_w, max(3, args.steps // 2), 3, dev, flush, stream)
            barrier()
        mla = None
        if main_w == I.PREFILL and not args.no_mla:
            mla = bench_mla(gdr, I.MLA_DECODE, max(3, args.steps // 2), 3, dev, stream)
            barrier()
        legs = {}
        if main_w == I.PREFILL and not args.no_long:
            for key, lw, k in (("long", I.LONG_PREFILL, max(3, args.steps // 2)),
                               ("million", I.MILLION_PREFILL, max(3, args.steps // 4))):
                legs[key] = bench_prefill_leg(gdr, lw, k, 3, dev, stream)
                barrier()
                if not (rank == 0 and world == 1 and not args.no_cpu_baseline):
                    legs[key] = (legs[key][0], None)   # the inputs are not needed any more
                torch.cuda.empty_cache()
    assert gdr.last_device_error(dev) == 0, "device error word set"

    ms_step = max_over_ranks(statistics.mean(ms))
    ms_e2e_step = max_over_ranks(statistics.mean(ms_e2e))
    if main_w.steps == 0:
        if varlen:   # the packed call takes the fused path chunk_fwd takes for B = S
            lengths = I.varlen_lengths(main_w)
            tokens = sum(lengths)
            by, fl = varlen_algorithmic(main_w, lengths)
        else:
            tokens = main_w.B * main_w.T
            by, fl = prefill_algorithmic(main_w)
        nk = gdr.chunk_fwd_kernels(main_w.B, main_w.H, main_w.T, main_w.dk, main_w.dv,
                                   main_w.chunk, main_w.a_min, main_w.torch_dtype())
        path = gdr.chunk_fwd_path(main_w.B, main_w.H, main_w.T, main_w.dk, main_w.dv,
                                  main_w.chunk, main_w.a_min, main_w.torch_dtype(),
                                  workspace=not args.single_launch)
        assert not varlen or path in (2, 3, 4, 5), "the packed call runs the fused or two-kernel path"
        kname, srcs, nk = path_kernels(path)
        metric = "packed prefill tokens/s" if varlen else "prefill tokens/s"
    else:
        tokens = main_w.B
        by, fl = decode_algorithmic(main_w), 0
        nk = 1
        kname = "decode128_kernel"
        srcs = ["gated_delta_rule_gdr_gb300/csrc/gdr_decode.cu"]
        metric = "decode tokens/s"
    value = world * tokens / (ms_step * 1e-3)
    achieved_gbs = by / (statistics.mean(ms) * 1e-3) / 1e9
    achieved_tf = fl / (statistics.mean(ms) * 1e-3) / 1e12
    t_roof = max(by / (pk["hbm_gbs"] * 1e9), fl / (pk["bf16_tflops"] * 1e12))
    bound = "hbm" if by / (pk["hbm_gbs"] * 1e9) >= fl / (pk["bf16_tflops"] * 1e12) else "tensor"
    roof = {
        "bound": bound, "kernel": kname,
        "achieved": round(achieved_gbs if bound == "hbm" else achieved_tf, 2),
        "peak": pk["hbm_gbs"] if bound == "hbm" else pk["bf16_tflops"],
        "peak_kind": pk_kind,
        "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
        "frac": None, "traffic": committed_traffic(kname, srcs, main_w.name),
        "algorithmic_bytes": by, "algorithmic_flops": fl,
        "frac_of_roofline_time": round(t_roof / (statistics.mean(ms) * 1e-3), 4),
        "achieved_tflops": round(achieved_tf, 2),
        "nominal_hbm_frac": round(achieved_gbs / 7900.0, 4),
    }
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    line = {
        "metric": metric, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": main_w.dtype, "data": "synthetic (seeded; recipe in gated_delta_rule_gdr_gb300/inputs.py)",
        "config": {"workload": main_w.name, "B": main_w.B, "H": main_w.H, "T": main_w.T,
                   "dk": main_w.dk, "dv": main_w.dv, "chunk": main_w.chunk,
                   **({"total_T": tokens} if varlen else {}),
                   "a_min": main_w.a_min, "parallelism": f"replicas x{world}",
                   "l2": "256 MB L2 flush between timed steps" if main_w.steps == 0
                   else "state (537 MB) larger than L2, no flush"},
        "roofline": roof,
        "e2e": {"value": round(world * tokens / (ms_e2e_step * 1e-3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(ms_e2e_step, 4),
                **({"api": "gdr_chunk_fwd_host (host buffers), two streams and device buffers "
                           "alternating"} if (main_w.steps == 0 and not varlen) else {})},
        "gpu_launches": nk * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed_region": round(wall, 3),
        "ms_per_step_all": [round(t, 4) for t in ms],
    }
    if dec is not None:
        dms, dms_e2e, dh2d, dd2h = dec
        w4 = I.DECODE
        dby = decode_algorithmic(w4)
        dmean = statistics.mean(dms)
        dgbs = dby / (dmean * 1e-3) / 1e9
        line["decode"] = {
            "metric": "decode tokens/s", "workload": w4.name,
            "value": round(world * w4.B / (max_over_ranks(dmean) * 1e-3), 1),
            "unit": "tokens/s", "ms_per_step": round(dmean, 4), "steps": args.decode_steps,
            "roofline": {"bound": "hbm", "kernel": "decode128_kernel", "achieved": round(dgbs, 1),
                         "peak": pk["hbm_gbs"], "peak_kind": pk_kind, "unit": "GB/s",
                         "frac": round(dgbs / pk["hbm_gbs"], 4),
                         "traffic": committed_traffic("decode128_kernel", [CSRC + "gdr_decode.cu"]),
                         "algorithmic_bytes": dby, "nominal_hbm_frac": round(dgbs / 7900.0, 4)},
            "e2e": {"value": round(world * w4.B / (max_over_ranks(statistics.mean(dms_e2e)) * 1e-3), 1),
                    "unit": "tokens/s", "h2d_bytes_per_step": dh2d, "d2h_bytes_per_step": dd2h},
            "gpu_launches": args.decode_steps,
        }
    if bwd is not None:
        bms, bws = bwd
        bmean = statistics.mean(bms)
        bby = backward_algorithmic(main_w)
        bgbs = bby / (bmean * 1e-3) / 1e9
        line["backward"] = {
            "metric": "backward tokens/s", "workload": main_w.name,
            "value": round(world * main_w.B * main_w.T / (max_over_ranks(bmean) * 1e-3), 1),
            "unit": "tokens/s", "ms_per_step": round(bmean, 4), "steps": len(bms),
            "roofline": {"bound": "hbm", "kernel": BWD_KERNELS, "achieved": round(bgbs, 1),
                         "peak": pk["hbm_gbs"], "peak_kind": pk_kind, "unit": "GB/s",
                         "frac": round(bgbs / pk["hbm_gbs"], 4),
                         "traffic": committed_traffic(BWD_KERNELS, BWD_SRCS + _COMMON + [CSRC + "gdr_prep.cu",
                                                                                       CSRC + "gdr_chain.cu"],
                                                      main_w.name),
                         "algorithmic_bytes": bby},
            "workspace_bytes": bws, "gpu_launches": 4 * len(bms),
        }
    if train is not None:
        tms, tfm, tbm, tsv, tnk = train
        tmean = statistics.mean(tms)
        tby = prefill_algorithmic(main_w)[0] + backward_algorithmic(main_w)
        tgbs = tby / (tmean * 1e-3) / 1e9
        line["training"] = {
            "metric": "training tokens/s", "workload": main_w.name,
            "what": "forward saving its chunk states + backward reading them, per step",
            "value": round(world * main_w.B * main_w.T / (max_over_ranks(tmean) * 1e-3), 1),
            "unit": "tokens/s", "ms_per_step": round(tmean, 4), "steps": len(tms),
            "forward_ms": round(statistics.mean(tfm), 4),
            "backward_ms": round(statistics.mean(tbm), 4),
            "roofline": {"bound": "hbm", "kernel": TRAIN_KERNELS, "achieved": round(tgbs, 1),
                         "peak": pk["hbm_gbs"], "peak_kind": pk_kind, "unit": "GB/s",
                         "frac": round(tgbs / pk["hbm_gbs"], 4), "algorithmic_bytes": tby,
                         "traffic": committed_traffic(TRAIN_KERNELS,
                                                      BWD_SRCS + _COMMON + [CSRC + "gdr_prep.cu",
                                                                            CSRC + "gdr_chain.cu"],
                                                      main_w.name)},
            "saved_bytes": tsv, "gpu_launches": tnk * len(tms),
        }
    if mla is not None:
        wm = I.MLA_DECODE
        mms, _ = mla
        mmean = statistics.mean(mms)
        mby, mfl = mla_algorithmic(wm)
        mgbs = mby / (mmean * 1e-3) / 1e9
        line["mla"] = {
            "metric": "latent-attention decode tokens/s", "workload": wm.name,
            "value": round(world * wm.N / (max_over_ranks(mmean) * 1e-3), 1), "unit": "tokens/s",
            "ms_per_step": round(mmean, 4), "steps": len(mms),
            "roofline": {"bound": "hbm", "kernel": "mla_attn_kernel + mla_combine_kernel",
                         "achieved": round(mgbs, 1), "peak": pk["hbm_gbs"], "peak_kind": pk_kind,
                         "unit": "GB/s", "frac": round(mgbs / pk["hbm_gbs"], 4),
                         "traffic": committed_traffic("mla_attn_kernel + mla_combine_kernel",
                                                      [CSRC + "gdr_mla.cu"] + _COMMON, wm.name),
                         "algorithmic_bytes": mby, "algorithmic_flops": mfl,
                         "achieved_tflops": round(mfl / (mmean * 1e-3) / 1e12, 2),
                         "tensor_frac": round(mfl / (mmean * 1e-3) / 1e12 / pk["bf16_tflops"], 4)},
            "l2": "cache (1 GiB) larger than L2, no flush",
            "gpu_launches": 2 * len(mms),
            "ms_per_step_all": [round(t, 4) for t in mms],
        }
    for key, (lms, _) in legs.items():
        line[key] = prefill_leg_line(gdr, {"long": I.LONG_PREFILL, "million": I.MILLION_PREFILL}[key],
                                     lms, pk, pk_kind, world, max_over_ranks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = (cpu_baseline_varlen(main_w) if varlen
                                else cpu_baseline_prefill(main_w) if main_w.steps == 0
                                else cpu_baseline_decode(main_w))
        if dec is not None:
            line["decode"]["cpu_baseline"] = cpu_baseline_decode(I.DECODE)
        if bwd is not None:
            line["backward"]["cpu_baseline"] = cpu_baseline_backward(main_w)
        if mla is not None:
            line["mla"]["cpu_baseline"] = cpu_baseline_mla(I.MLA_DECODE, mla[1])
            mla = None
        for key, (_, lx) in legs.items():
            lw = {"long": I.LONG_PREFILL, "million": I.MILLION_PREFILL}[key]
            line[key]["cpu_baseline"] = cpu_baseline_prefill(lw, budget_s=6.0, x=lx)
            legs[key] = None
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


WORKLOAD_ARG = {"prefill": I.PREFILL, "long": I.LONG_PREFILL, "million": I.MILLION_PREFILL,
                "decode": I.DECODE, "varlen": I.VARLEN}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    """The fp64 CPU oracle, as it stands, on bounded samples of the workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    w = WORKLOAD_ARG[args.workload]
    cores = os.cpu_count() or 1
    times = []
    if w is I.VARLEN:
        lengths = I.varlen_lengths(w)
        toks = []
        for i in range(args.warmup + args.steps):
            tok, dt, n = oracle_varlen_sample(w, lengths, 2.0, cores)
            if i >= args.warmup:
                times.append(dt)
                toks.append(tok)
        tok = statistics.mean(toks)
        sample = f"per step: the first {n} of {len(lengths)} sequences, all {w.H} heads ({tok} tokens)"
        metric = "packed prefill tokens/s"
    elif w.steps == 0:
        x = I.prefill_inputs(w.with_(B=1), device="cpu")
        Ts = min(w.T, 512)
        sub = {n: x[n][:, :, :Ts] for n in ("q", "k", "v", "g", "beta")}
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            oracle.fwd(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], w.a_min,
                       x["init_state"], nthreads=cores)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
        tok = Ts                     # B*T-tokens of the workload processed per step
        sample = f"per step: B=1, all {w.H} heads, first {Ts} of {w.T} tokens"
        metric = "prefill tokens/s"
    else:
        state = I.decode_state(w, device="cpu").double().numpy().copy()
        for i in range(args.warmup + args.steps):
            x = I.decode_step_inputs(w, i % w.steps, device="cpu")
            t0 = time.perf_counter()
            oracle.decode(x["q"], x["k"], x["v"], x["g"], x["beta"], w.a_min, state,
                          nthreads=cores)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
        tok = w.B
        sample = f"per step: one decode step over all {w.B}x{w.H} (n,h)"
        metric = "decode tokens/s"
    mean = statistics.mean(times)
    value = tok / mean
    line = {"impl": "reference", "metric": metric, "value": round(value, 2), "unit": "tokens/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(mean * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "dk": w.dk, "dv": w.dv,
                       "chunk": w.chunk, "a_min": w.a_min},
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--decode-steps", type=int, default=64)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_ARG),
                    default="prefill")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-mla", action="store_true",
                    help="skip the gated latent-attention decode leg")
    ap.add_argument("--no-long", action="store_true",
                    help="skip the long (B1 H32 T65536) and million-token (B1 H16 T1048576) legs")
    ap.add_argument("--B", type=int, default=0, help="override B of a prefill workload (profiling)")
    ap.add_argument("--H", type=int, default=0, help="override H of a prefill workload (profiling)")
    ap.add_argument("--T", type=int, default=0, help="override T of a prefill workload (profiling)")
    ap.add_argument("--single-launch", action="store_true",
                    help="the one-launch fused path (no workspace) instead of prep + chain")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
