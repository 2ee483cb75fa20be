#!/usr/bin/env python3
"""Throughput of the liboss hot path on one GB300 (or N, one process each).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload (``config.workload``): softmax_32k -- os_softmax_rows over a
32768 x 8192 fp32 matrix of N(0,1) * 10 logits (1 GiB in, 1 GiB out). A step
is one os_softmax_rows call; ``value`` is algorithmic GB/s (bytes read + bytes
written by the definition) over all ranks. The same JSON line carries, under
``extra``, the two- and three-pass comparators on the same matrix (value in
the same algorithmic GB/s, so the ratio is the saving of the one-pass form),
the same matrix stored in bf16 (softmax_32k_bf16), the attention forward (attn_4k, non-causal; attn_causal) in
TFLOP/s and split-KV decode + merge (decode_64x32) in GB/s, each with its own
roofline.

Inputs are seeded and synthetic, resident in HBM before the timed region, and
larger than the 129 MB L2 (no flush needed). Timing: W untimed steps, then K
steps bracketed by a barrier and a device synchronise, CUDA events on the
launching stream, max over ranks. ``--impl reference`` times the fp64 CPU
oracle on the host cores on bounded samples of the same workload.
"""

from __future__ import annotations

import argparse
import collections
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from pass_attention_gb300 import workloads  # noqa: E402

METRIC = "softmax GB/s & attention fwd TFLOP/s on 1 GB300, as fraction of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# the GB300's nominal figures, reported beside the measured-peak fractions
NOMINAL = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0}

# DRAM traffic per launch from ncu (dram__bytes_read.sum + dram__bytes_write.sum),
# keyed by workload, with the sha256 of the kernel source's code (comments and
# blank lines removed) when it was captured: changed code reports null. Summaries live under profiles/.
# "scale" records traffic / algorithmic bytes of a smaller capture of the
# same kernel, applied to the full launch's algorithmic bytes.
_SRC_COMMON = ["pass_attention_gb300/csrc/softmax_common.cuh",
               "pass_attention_gb300/csrc/device_common.cuh"]
_SRC_ROWS = ["pass_attention_gb300/csrc/softmax_rows.cu"] + _SRC_COMMON
_SRC_GROUPED = ["pass_attention_gb300/csrc/softmax_grouped.cu"] + _SRC_COMMON
_SRC_WIDE = ["pass_attention_gb300/csrc/softmax_wide.cu"] + _SRC_COMMON
NCU_TRAFFIC = {
    "softmax_32k": {"source": _SRC_ROWS,
                    "sha256": "73995524e85db31d7c3bf8d58cf01f5782d07ad3a36db8fe5429e33fcd182570",
                    "bytes_per_launch": 1073778688 + 1017928448},
    "softmax_32k_bf16": {"source": _SRC_GROUPED,
                         "sha256": "edca4d93214216b2621d11a822fc211291dd35ffdef21c5c7f9f9b25c782109f",
                         "bytes_per_launch": 536895488 + 484645376},
    # the comparators: all sweeps of one call (each reads x from DRAM again)
    "softmax_32k_3pass": {"source": _SRC_ROWS,
                          "sha256": "73995524e85db31d7c3bf8d58cf01f5782d07ad3a36db8fe5429e33fcd182570",
                          "bytes_per_launch": (1073760768 + 2916608) + (1073907712 + 246528)
                          + (1074052608 + 1024674048)},
    "softmax_32k_2pass": {"source": _SRC_ROWS,
                          "sha256": "73995524e85db31d7c3bf8d58cf01f5782d07ad3a36db8fe5429e33fcd182570",
                          "bytes_per_launch": (1073760000 + 2976000) + (1074086656 + 1024858624)},
    # rows over 1.6 MB, the cooperative kernel (one read from HBM, one from L2)
    "softmax_64x4m_fp32": {"source": _SRC_WIDE,
                           "sha256": "9abfeac38fb9931ea4f304e1c199c04d026e43d90bd0e247fea097ca74f14fc8",
                           "bytes_per_launch": 1289380608 + 1013640960},
    "softmax_64x4m_bf16": {"source": _SRC_WIDE,
                           "sha256": "9abfeac38fb9931ea4f304e1c199c04d026e43d90bd0e247fea097ca74f14fc8",
                           "bytes_per_launch": 633526272 + 478089472},
    "attn_4k": {"source": "pass_attention_gb300/csrc/attn_fwd.cu",
                "sha256": "1be6e0f202facc625839827f2a87382ddd1d773a7096bf3895c42b0e52cfff77",
                "bytes_per_launch": 201534464 + 49693952},
    "attn_causal": {"source": "pass_attention_gb300/csrc/attn_fwd.cu",
                    "sha256": "1be6e0f202facc625839827f2a87382ddd1d773a7096bf3895c42b0e52cfff77",
                    "bytes_per_launch": 405638400 + 119282688},
    "decode_64x32": {"source": "pass_attention_gb300/csrc/decode_merge.cu",
                     "sha256": "0d345bb183c174c3248d68638b3899f9499e35b1a5ceb04884c68dbc28755393",
                     # B 8, H 32, Lmax 8192 (kv_len sum 36965), 16 splits
                     "scale": (605719552 + 3959040) / (36965 * 32 * 512 + 8 * 32 * 128 * 2
                                                       + 8 * 32 * 16 * 130 * 4)},
}


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def source_sha(rel):
    """sha256 of a kernel's sources (one path, or a list: the kernel's file and
    the headers it includes) with comments and blank lines removed, so that a
    comment edit keeps the ncu figures taken of the same code."""
    import re
    h = hashlib.sha256()
    for path in ([rel] if isinstance(rel, str) else rel):
        with open(os.path.join(ROOT, path)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
        h.update("\n".join(ln for ln in lines if ln.strip()).encode())
    return h.hexdigest()


def traffic_for(workload, algorithmic_bytes=None):
    rec = NCU_TRAFFIC.get(workload)
    if not rec:
        return None
    try:
        if source_sha(rec["source"]) != rec["sha256"]:
            return None
    except OSError:
        return None
    if "scale" in rec:
        return None if algorithmic_bytes is None else rec["scale"] * algorithmic_bytes
    return rec["bytes_per_launch"]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ["timestamp", "index", "clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        inside = [p for (t, p) in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        window = "timed region"
        if not inside:
            inside = [p for (_, p) in self.samples]
            window = "whole run (timed region shorter than the 100 ms sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        sm = [float(p[2]) for p in inside if p[2].replace(".", "").isdigit()]
        smax = [float(p[3]) for p in inside if p[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(inside), "window": window}


def device_index_for_smi(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids) and ids[local_rank].isdigit():
            return int(ids[local_rank])
    return local_rank


Timing = collections.namedtuple("Timing", "total_ms mean_ms median_ms t0 t1")


def headline_config(w):
    """The headline's ``config`` dict, shared by both arms so that their lines
    name the same workload in the same words."""
    return {"workload": f"{w.name} {w.rows}x{w.cols} fp32 N(0,1)*{w.mult:g}, scale {w.scale:g}",
            "rows": w.rows, "cols": w.cols, "per_rank": "one full matrix per rank",
            "l2": "inputs larger than L2 (1 GiB per step), no flush"}


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise maximum of per-rank timings over all ranks (the slowest
    rank decides a step's time). ``dist`` is torch.distributed or None for a
    single process; ``device`` is where the collective's tensor lives (cuda
    for NCCL, cpu for gloo)."""
    values = [float(v) for v in values]
    if dist is None:
        return values
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def time_steps(fn, steps, warmup, stream, barrier):
    """W untimed calls, then K timed calls with per-step events. Returns a
    Timing: the K-step total, the mean and median step (ms), and the wall
    clock at both ends."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    t0 = time.time()
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(steps):
            fn()
            ev[i + 1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    return Timing(ev[0].elapsed_time(ev[steps]), sum(per) / len(per), statistics.median(per), t0, t1)


# ---------------------------------------------------------------------------
# workloads on the GPU
# ---------------------------------------------------------------------------

def softmax_bytes(rows, cols):
    return rows * cols * 4 * 2 + rows * 4 * 2  # x read, y written, m and l written


def attention_flops(B, H, S, D, causal):
    if causal:
        return 4 * B * H * D * (S * (S + 1) // 2)
    return 4 * B * H * S * S * D


def decode_bytes(kv_len, H, D, S):
    B = len(kv_len)
    kv = int(sum(int(L) for L in kv_len)) * H * D * 2 * 2   # K and V rows read once
    q = B * H * D * 2
    parts = B * H * S * (D + 2) * 4                         # written by decode, read by merge
    out = B * H * (D * 2 + 4 * 3)                           # O bf16, m, l, lse
    return kv + q + 2 * parts + out


def bench_softmax(args, ctx):
    import pass_attention_gb300 as oss
    w = workloads.SOFTMAX_32K
    x = workloads.logits(w.rows, w.cols, w.mult, w.seed + ctx["rank"], device="cuda")
    y = torch.empty_like(x)
    m = torch.empty(w.rows, device="cuda")
    l = torch.empty(w.rows, device="cuda")
    stream = torch.cuda.current_stream()
    fn = lambda: oss.softmax_rows(x, w.scale, y=y, m=m, l=l, stream=stream)
    total_ms, step_ms, median_ms, t0, t1 = time_steps(fn, args.steps, args.warmup, stream,
                                                      ctx["barrier"])
    nbytes = softmax_bytes(w.rows, w.cols)
    # end to end: pinned host input -> device -> kernel -> pinned host outputs
    xh = x.cpu().pin_memory()
    outs = (torch.empty(x.shape, pin_memory=True), torch.empty(w.rows, pin_memory=True),
            torch.empty(w.rows, pin_memory=True))
    e2e_steps = max(1, min(args.steps, 10))
    oss.softmax_rows_from_host(xh, w.scale, out=outs, x_dev=x, y_dev=y)
    torch.cuda.synchronize()
    ctx["barrier"]()
    # three timed blocks of e2e_steps calls; the median block is reported (a
    # block that meets contention on the shared host side does not decide it)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    blocks = []
    for _ in range(3):
        s.record()
        for _ in range(e2e_steps):
            oss.softmax_rows_from_host(xh, w.scale, out=outs, x_dev=x, y_dev=y)
        e.record()
        torch.cuda.synchronize()
        blocks.append(s.elapsed_time(e) / e2e_steps)
    e2e_ms = statistics.median(blocks)
    # the host link on this machine: plain pinned copies of the same buffers, both
    # directions at once (the e2e step cannot beat this)
    s_up, s_dn = torch.cuda.Stream(), torch.cuda.Stream()

    def both():
        with torch.cuda.stream(s_up):
            x.copy_(xh, non_blocking=True)
        with torch.cuda.stream(s_dn):
            outs[0].copy_(y, non_blocking=True)

    both()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    s.record()
    for _ in range(5):
        s_up.wait_stream(cur)
        s_dn.wait_stream(cur)
        both()
        cur.wait_stream(s_up)
        cur.wait_stream(s_dn)
    e.record()
    torch.cuda.synchronize()
    link_gbs = 2 * w.rows * w.cols * 4 * 5 / (s.elapsed_time(e) / 1e3) / 1e9
    del xh, outs
    return {"workload": w, "total_ms": total_ms, "step_ms": step_ms, "median_ms": median_ms,
            "t0": t0, "t1": t1,
            "nbytes": nbytes, "e2e_ms": e2e_ms, "e2e_blocks_ms": blocks, "link_gbs": link_gbs,
            "h2d": w.rows * w.cols * 4,
            "d2h": w.rows * w.cols * 4 + 2 * w.rows * 4}


def bench_softmax_multipass(args, ctx, passes):
    """The comparators of os_softmax_rows on the same matrix: the safe
    softmax's three sweeps (max, sum, write) or the online normaliser followed
    by a write sweep. Returns (ms per call, HBM bytes the sweeps move)."""
    import pass_attention_gb300 as oss
    w = workloads.SOFTMAX_32K
    x = workloads.logits(w.rows, w.cols, w.mult, w.seed + ctx["rank"], device="cuda")
    y = torch.empty_like(x)
    m = torch.empty(w.rows, device="cuda")
    l = torch.empty(w.rows, device="cuda")
    stream = torch.cuda.current_stream()
    fn = lambda: oss.softmax_rows_multipass(x, passes, w.scale, y=y, m=m, l=l, stream=stream)
    steps = max(3, min(args.steps, 30))
    tm = time_steps(fn, steps, max(3, args.warmup), stream, ctx["barrier"])
    moved = w.rows * w.cols * 4 * (passes + 1) + w.rows * 4 * (2 * passes + 2)
    return tm, moved


def bench_softmax16(args, ctx):
    """os_softmax_rows_16bit on the softmax_32k matrix stored in bf16."""
    import pass_attention_gb300 as oss
    w = workloads.SOFTMAX_32K
    x = workloads.logits(w.rows, w.cols, w.mult, w.seed + ctx["rank"],
                         device="cuda").to(torch.bfloat16)
    y = torch.empty_like(x)
    m = torch.empty(w.rows, device="cuda")
    l = torch.empty(w.rows, device="cuda")
    stream = torch.cuda.current_stream()
    fn = lambda: oss.softmax_rows_16bit(x, w.scale, y=y, m=m, l=l, stream=stream)
    steps = max(3, min(args.steps, 50))
    tm = time_steps(fn, steps, max(3, args.warmup), stream, ctx["barrier"])
    nbytes = w.rows * w.cols * 2 * 2 + w.rows * 4 * 2
    return tm, nbytes


def bench_softmax_long(args, ctx):
    """Rows beyond a cluster's shared memory: 64 x 2^22 fp32 (16 MB rows,
    1 GiB) and the same matrix in bf16, through os_softmax_rows_ws /
    os_softmax_rows_16bit_ws (the binding supplies the workspace). Returns
    {name: (Timing, algorithmic bytes)}."""
    import pass_attention_gb300 as oss
    out = {}
    stream = torch.cuda.current_stream()
    rows, cols = 64, 1 << 22
    for name, dtype in (("fp32", torch.float32), ("bf16", torch.bfloat16)):
        x = workloads.logits(rows, cols, 10.0, 11 + ctx["rank"], device="cuda").to(dtype)
        y = torch.empty_like(x)
        m = torch.empty(rows, device="cuda")
        l = torch.empty(rows, device="cuda")
        if dtype == torch.float32:
            fn = lambda: oss.softmax_rows(x, 1.0, y=y, m=m, l=l, stream=stream)
        else:
            fn = lambda: oss.softmax_rows_16bit(x, 1.0, y=y, m=m, l=l, stream=stream)
        tm = time_steps(fn, max(3, min(args.steps, 20)), 3, stream, ctx["barrier"])
        out[name] = (tm, rows * cols * 2 * x.element_size() + rows * 8)
        del x, y
    return out


def bench_softmax_lengths(args, ctx):
    """os_softmax_rows / os_softmax_rows_16bit over row lengths from 128 to
    131072 at 2^28 elements per matrix (1 GiB fp32, 512 MiB 16-bit: larger
    than L2). Returns {dtype: {cols: (ms per call, algorithmic bytes)}}."""
    import pass_attention_gb300 as oss
    out = {}
    stream = torch.cuda.current_stream()
    for name, dtype in (("fp32", torch.float32), ("bf16", torch.bfloat16), ("fp16", torch.float16)):
        out[name] = {}
        for cols in (128, 512, 1024, 2048, 4096, 8192, 16384, 32768, 131072):
            rows = (1 << 28) // cols
            x = workloads.logits(rows, cols, 10.0, 7 + ctx["rank"], device="cuda").to(dtype)
            y = torch.empty_like(x)
            m = torch.empty(rows, device="cuda")
            l = torch.empty(rows, device="cuda")
            if dtype == torch.float32:
                fn = lambda: oss.softmax_rows(x, 1.0, y=y, m=m, l=l, stream=stream)
            else:
                fn = lambda: oss.softmax_rows_16bit(x, 1.0, y=y, m=m, l=l, stream=stream)
            tm = time_steps(fn, 10, 3, stream, ctx["barrier"])
            out[name][cols] = (tm.mean_ms, rows * cols * 2 * x.element_size() + rows * 8)
            del x, y
    return out


def bench_attention(args, ctx, w):
    import pass_attention_gb300 as oss
    q, k, v = workloads.qkv(w.B, w.H, w.S, w.S, w.D, w.seed, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), device="cuda")
    stream = torch.cuda.current_stream()
    fn = lambda: oss.attention_fwd(q, k, v, w.scale, w.causal, o=o, lse=lse, stream=stream)
    steps = max(3, min(args.steps, 50))
    tm = time_steps(fn, steps, max(3, args.warmup), stream, ctx["barrier"])
    oss.check_device_error()
    flops = attention_flops(w.B, w.H, w.S, w.D, w.causal)
    cpu = None
    if ctx["rank"] == 0 and args.extra_cpu_seconds > 0:
        rate, cores, rows, full_s = oracle_attention_rate(q, k, v, w, args.extra_cpu_seconds)
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{rows} seeded query rows of 4 heads, 64 at a time, "
                         f"~{args.extra_cpu_seconds:g} s on {cores} host threads",
               "extrapolated_full_s": full_s}
    return tm, flops, cpu


def bench_decode(args, ctx):
    import pass_attention_gb300 as oss
    w = workloads.DECODE_64X32
    q, k, v, kv = workloads.decode_inputs(w.B, w.H, w.Lmax, w.D, w.seed, device="cuda")
    S = w.num_splits
    pm = torch.empty((w.B, w.H, S), device="cuda")
    pl = torch.empty_like(pm)
    po = torch.empty((w.B, w.H, S, w.D), device="cuda")
    o = torch.empty((w.B, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    mo, lo, lseo = (torch.empty((w.B, w.H), device="cuda") for _ in range(3))
    stream = torch.cuda.current_stream()

    def fn():
        oss.attention_decode_splitkv(q, k, v, kv, S, w.scale, pm, pl, po, stream=stream)
        oss.merge_partials(pm, pl, po, True, o, mo, lo, lseo, stream=stream)

    steps = max(3, min(args.steps, 30))
    tm = time_steps(fn, steps, max(3, args.warmup), stream, ctx["barrier"])
    # the decode kernel alone (dominant): events around it only
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps)]
    for i in range(steps):
        ev[2 * i].record(stream)
        oss.attention_decode_splitkv(q, k, v, kv, S, w.scale, pm, pl, po, stream=stream)
        ev[2 * i + 1].record(stream)
    torch.cuda.synchronize()
    dec_ms = sum(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(steps)) / steps
    kvl = kv.cpu().tolist()
    nbytes = decode_bytes(kvl, w.H, w.D, S)
    kv_bytes = int(sum(kvl)) * w.H * w.D * 4
    dec_bytes = kv_bytes + w.B * w.H * w.D * 2 + w.B * w.H * S * (w.D + 2) * 4
    cpu = None
    if ctx["rank"] == 0 and args.extra_cpu_seconds > 0:
        rate, cores, rows = oracle_decode_rate(q, k, v, kv, w, args.extra_cpu_seconds)
        cpu = {"value": rate, "unit": "GB/s (K and V read)", "cores": cores, "kind": "oracle",
               "sample": f"{rows} seeded (b, h) query rows over their whole kv_len, "
                         f"~{args.extra_cpu_seconds:g} s on {cores} host threads"}
    del k, v
    return tm, nbytes, dec_ms, dec_bytes, cpu


# ---------------------------------------------------------------------------
# the oracle on the host cores
# ---------------------------------------------------------------------------

def oracle_softmax_rate(seconds, x_np=None):
    """Time the fp64 oracle's softmax on row chunks of the softmax_32k
    workload across the host cores (numpy releases the GIL in its ufuncs)
    until about ``seconds`` have passed. Returns (GB/s, cores, rows)."""
    import oracle
    w = workloads.SOFTMAX_32K
    chunk = 256
    if x_np is None:
        x_np = workloads.logits(4096, w.cols, w.mult, w.seed).numpy()
    cores = os.cpu_count() or 1
    done_rows = 0
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=cores) as ex:
        while time.perf_counter() - t0 < seconds:
            starts = [(i * chunk) % x_np.shape[0] for i in range(cores)]
            list(ex.map(lambda s: oracle.softmax_rows(x_np[s:s + chunk], w.scale), starts))
            done_rows += chunk * cores
    dt = time.perf_counter() - t0
    return softmax_bytes(done_rows, w.cols) / dt / 1e9, cores, done_rows


def oracle_attention_rate(q, k, v, w, seconds):
    """Time the fp64 oracle's attention on seeded sample rows of an attention
    workload (64 query rows at a time, from four heads) on the host cores for
    about ``seconds``. Returns (TFLOP/s, cores, rows, extrapolated seconds for
    the whole workload)."""
    import oracle
    rng = np.random.default_rng(w.seed)
    heads = [(int(rng.integers(w.B)), int(rng.integers(w.H))) for _ in range(4)]
    host = {bh: tuple(t[bh[0]:bh[0] + 1, bh[1]:bh[1] + 1].float().cpu().numpy().astype(np.float64)
                      for t in (q, k, v)) for bh in heads}
    cores = os.cpu_count() or 1

    def job(i):
        qh, kh, vh = host[heads[i % len(heads)]]
        rows = [(0, 0, (i * 977 + j * 61) % w.S) for j in range(64)]
        oracle.attention(qh, kh, vh, w.scale, w.causal, rows=rows)
        return sum(4 * w.D * ((r[2] + 1) if w.causal else w.S) for r in rows)

    flops, n = 0, 0
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=cores) as ex:
        while time.perf_counter() - t0 < seconds:
            flops += sum(ex.map(job, range(n, n + cores)))
            n += cores
    dt = time.perf_counter() - t0
    rate = flops / dt / 1e12
    return rate, cores, n * 64, attention_flops(w.B, w.H, w.S, w.D, w.causal) / (rate * 1e12)


def oracle_decode_rate(q, k, v, kv, w, seconds):
    """Time the fp64 oracle's decode on seeded (b, h) rows of the decode
    workload on the host cores for about ``seconds``. Returns (GB/s of K and V
    read, cores, rows)."""
    import oracle
    rng = np.random.default_rng(w.seed)
    kvl = kv.cpu().numpy()
    pairs = [(int(rng.integers(w.B)), int(rng.integers(w.H))) for _ in range(8)]
    host = {}
    for b, h in pairs:
        L = int(kvl[b])
        host[(b, h)] = (q[b:b + 1, h:h + 1].float().cpu().numpy().astype(np.float64),
                        k[b:b + 1, h:h + 1, :L].float().cpu().numpy().astype(np.float64),
                        v[b:b + 1, h:h + 1, :L].float().cpu().numpy().astype(np.float64), L)
    cores = os.cpu_count() or 1

    def job(i):
        qh, kh, vh, L = host[pairs[i % len(pairs)]]
        oracle.decode(qh, kh, vh, np.array([L]), w.scale)
        return L * w.D * 2 * 2

    nbytes, n = 0, 0
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=cores) as ex:
        while time.perf_counter() - t0 < seconds:
            nbytes += sum(ex.map(job, range(n, n + cores)))
            n += cores
    dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, cores, n


def run_reference(args, rank):
    if rank != 0:
        return
    w = workloads.SOFTMAX_32K
    x_np = workloads.logits(4096, w.cols, w.mult, w.seed).numpy()
    per_step_s = args.ref_step_seconds
    for _ in range(args.warmup):
        oracle_softmax_rate(0.2, x_np)
    t0 = time.perf_counter()
    rates = []
    rows_total = 0
    for _ in range(args.steps):
        r, cores, rows = oracle_softmax_rate(per_step_s, x_np)
        rates.append(r)
        rows_total += rows
    dt = time.perf_counter() - t0
    value = softmax_bytes(rows_total, w.cols) / dt / 1e9
    sample = (f"{rows_total} rows of the {w.rows}x{w.cols} workload over {args.steps} steps "
              f"(~{per_step_s:.0f} s each), 256-row chunks on {cores} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": headline_config(w),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--extra-cpu-seconds", type=float, default=3.0,
                    help="oracle time beside each attention / decode extra (rank 0)")
    ap.add_argument("--ref-step-seconds", type=float, default=2.0,
                    help="oracle time per step of --impl reference")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend)

    if args.impl == "reference":
        run_reference(args, rank)
        if dist:
            dist.destroy_process_group()
        return

    import pass_attention_gb300 as oss
    oss.load()  # fails loudly if the library is not built
    torch.cuda.set_device(local_rank)

    def barrier():
        if dist:
            dist.barrier()

    ctx = {"rank": rank, "barrier": barrier}
    pk, pk_kind = peaks()
    sampler = ClockSampler(device_index_for_smi(local_rank)).start()

    sm = bench_softmax(args, ctx)
    total_ms = sm["total_ms"]
    step_ms = sm["step_ms"]
    e2e_ms = sm["e2e_ms"]
    total_ms, step_ms, e2e_ms = max_over_ranks([total_ms, step_ms, e2e_ms], dist, "cuda")
    n = world
    w = sm["workload"]
    value = sm["nbytes"] * args.steps * n / (total_ms / 1e3) / 1e9
    achieved = sm["nbytes"] / (sm["step_ms"] / 1e3) / 1e9
    kname = "softmax_rows_reg_kernel<8>"

    extra = {}
    if not args.headline_only:
        for passes in (3, 2):
            name = f"softmax_32k_{passes}pass"
            try:
                tm, moved = bench_softmax_multipass(args, ctx, passes)
                ms = tm.mean_ms
                moved_gbs = moved / (ms / 1e3) / 1e9
                extra[name] = {
                    "value": sm["nbytes"] / (ms / 1e3) / 1e9, "unit": "GB/s",
                    "ms_per_step": ms, "ms_per_step_median": tm.median_ms,
                    "one_pass_speedup": ms / sm["step_ms"],
                    "workload": f"{w.rows}x{w.cols} fp32, os_softmax_rows_multipass passes={passes}",
                    "hbm_bytes_per_step": moved,
                    "roofline": {"bound": "hbm", "achieved": moved_gbs, "peak": pk["hbm_gbs"],
                                 "unit": "GB/s", "frac": moved_gbs / pk["hbm_gbs"],
                                 "traffic": traffic_for(name), "peak_kind": f"{pk_kind} HBM copy",
                                 "nominal_peak": NOMINAL["hbm_gbs"],
                                 "frac_nominal": moved_gbs / NOMINAL["hbm_gbs"],
                                 "note": "achieved counts every sweep's bytes"},
                    "window": (tm.t0, tm.t1)}
            except Exception as e:
                extra[name] = {"unavailable": f"{type(e).__name__}: {e}"}
        try:
            tm, nbytes = bench_softmax16(args, ctx)
            ms = tm.mean_ms
            gbs = nbytes / (ms / 1e3) / 1e9
            extra["softmax_32k_bf16"] = {
                "value": gbs, "unit": "GB/s", "ms_per_step": ms, "ms_per_step_median": tm.median_ms,
                "workload": f"{w.rows}x{w.cols} bf16 rows (y bf16, m and l fp32), os_softmax_rows_16bit",
                "roofline": {"bound": "hbm",
                             "kernel": "softmax_rows_grouped_kernel<bf16, 256 threads a row, 4 chunks, 4 CTAs/SM>",
                             "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                             "frac": gbs / pk["hbm_gbs"], "traffic": traffic_for("softmax_32k_bf16"),
                             "peak_kind": f"{pk_kind} HBM copy", "nominal_peak": NOMINAL["hbm_gbs"],
                             "frac_nominal": gbs / NOMINAL["hbm_gbs"]},
                "window": (tm.t0, tm.t1)}
        except Exception as e:
            extra["softmax_32k_bf16"] = {"unavailable": f"{type(e).__name__}: {e}"}
        try:
            lens = bench_softmax_lengths(args, ctx)
            extra["softmax_row_lengths"] = {
                "unit": "GB/s",
                "workload": "2^28 elements per matrix, N(0,1)*10 logits, scale 1; cols 128..131072",
                "peak": pk["hbm_gbs"], "peak_kind": f"{pk_kind} HBM copy",
                "value": {d: {str(c): nb / (ms / 1e3) / 1e9 for c, (ms, nb) in v.items()}
                          for d, v in lens.items()},
                "frac": {d: {str(c): nb / (ms / 1e3) / 1e9 / pk["hbm_gbs"] for c, (ms, nb) in v.items()}
                         for d, v in lens.items()},
            }
        except Exception as e:
            extra["softmax_row_lengths"] = {"unavailable": f"{type(e).__name__}: {e}"}
        try:
            for name, (tm, nb) in bench_softmax_long(args, ctx).items():
                gbs = nb / (tm.mean_ms / 1e3) / 1e9
                extra[f"softmax_64x4m_{name}"] = {
                    "value": gbs, "unit": "GB/s", "ms_per_step": tm.mean_ms,
                    "ms_per_step_median": tm.median_ms,
                    "workload": f"64 x 2^22 {name} rows (16 MB fp32 / 8 MB bf16 a row), N(0,1)*10, "
                                "scale 1, with a workspace",
                    "roofline": {"bound": "hbm", "kernel": "softmax_rows_wide_kernel (cooperative)",
                                 "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                                 "frac": gbs / pk["hbm_gbs"], "traffic": traffic_for(f"softmax_64x4m_{name}"),
                                 "peak_kind": f"{pk_kind} HBM copy", "nominal_peak": NOMINAL["hbm_gbs"],
                                 "frac_nominal": gbs / NOMINAL["hbm_gbs"]},
                    "window": (tm.t0, tm.t1)}
        except Exception as e:
            extra["softmax_64x4m"] = {"unavailable": f"{type(e).__name__}: {e}"}
        for aw in (workloads.ATTN_4K, workloads.ATTN_CAUSAL):
            try:
                tm, flops, cpu_a = bench_attention(args, ctx, aw)
                ms = tm.mean_ms
                tf = flops / (ms / 1e3) / 1e12
                extra[aw.name] = {
                    "value": tf, "unit": "TFLOP/s", "ms_per_step": ms,
                    "ms_per_step_median": tm.median_ms,
                    "workload": f"B{aw.B} H{aw.H} S{aw.S} D{aw.D} bf16 {'causal' if aw.causal else 'non-causal'}",
                    "roofline": {"bound": "tensor", "achieved": tf, "peak": pk["bf16_tflops"],
                                 "unit": "TFLOP/s", "frac": tf / pk["bf16_tflops"],
                                 "traffic": traffic_for(aw.name),
                                 "peak_kind": f"{pk_kind} bf16 dense (burst)",
                                 "nominal_peak": NOMINAL["bf16_tflops"],
                                 "frac_nominal": tf / NOMINAL["bf16_tflops"]},
                    "cpu_baseline": cpu_a,
                    "window": (tm.t0, tm.t1)}
            except Exception as e:  # report, do not hide
                extra[aw.name] = {"unavailable": f"{type(e).__name__}: {e}"}
        try:
            tm, nbytes, dec_ms, dec_bytes, cpu_d = bench_decode(args, ctx)
            ms = tm.mean_ms
            gbs = nbytes / (ms / 1e3) / 1e9
            ach = dec_bytes / (dec_ms / 1e3) / 1e9
            extra["decode_64x32"] = {
                "value": gbs, "unit": "GB/s", "ms_per_step": ms, "ms_per_step_median": tm.median_ms,
                "workload": "B64 H32 D128 bf16, kv_len~U{1..32768}, 16 splits, decode + merge",
                "roofline": {"bound": "hbm", "kernel": "decode_splitkv_kernel", "achieved": ach,
                             "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": ach / pk["hbm_gbs"],
                             "traffic": traffic_for("decode_64x32", dec_bytes),
                             "peak_kind": f"{pk_kind} HBM copy",
                             "nominal_peak": NOMINAL["hbm_gbs"],
                             "frac_nominal": ach / NOMINAL["hbm_gbs"]},
                "cpu_baseline": cpu_d,
                "window": (tm.t0, tm.t1)}
        except Exception as e:
            extra["decode_64x32"] = {"unavailable": f"{type(e).__name__}: {e}"}

    sampler.stop()
    clocks = sampler.summary(sm["t0"], sm["t1"])
    for entry in extra.values():
        if "window" in entry:
            entry["clocks"] = sampler.summary(*entry.pop("window"))

    cpu = None
    if rank == 0:
        rate, cores, rows = oracle_softmax_rate(args.cpu_seconds)
        cpu = {"value": rate, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{rows} rows of the {w.rows}x{w.cols} workload in 256-row chunks, "
                         f"~{args.cpu_seconds:g} s on {cores} host threads"}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "ms_per_step_median": sm["median_ms"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": headline_config(w),
        "clocks": clocks,
        "e2e": {"value": sm["nbytes"] * n / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": sm["h2d"], "d2h_bytes_per_step": sm["d2h"],
                "host_link_gbs": sm["link_gbs"],
                "frac_of_host_link": (sm["nbytes"] / (e2e_ms / 1e3) / 1e9) / sm["link_gbs"],
                "blocks_gbs": [sm["nbytes"] / (b / 1e3) / 1e9 for b in sm["e2e_blocks_ms"]],
                "note": "median of three timed blocks of calls (blocks_gbs); host_link_gbs: "
                        "pinned H2D + D2H copies of the same buffers, both at once"},
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                     "traffic": traffic_for(w.name), "peak_kind": f"{pk_kind} HBM copy",
                     "nominal_peak": NOMINAL["hbm_gbs"],
                     "frac_nominal": achieved / NOMINAL["hbm_gbs"]},
        "cpu_baseline": cpu,
        "extra": extra,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
