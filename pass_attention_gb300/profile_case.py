"""Run one liboss entry point on one workload a few times, for profilers.

    python -m pass_attention_gb300.profile_case softmax [--rows R --cols C] [--reps N] [--no-ws]
    python -m pass_attention_gb300.profile_case softmax16 [--dtype bf16|f16] [--rows R --cols C] [--no-ws]
    python -m pass_attention_gb300.profile_case multipass --passes 2|3 [--rows R --cols C]
    python -m pass_attention_gb300.profile_case attn [--B --H --S] [--causal] [--reps N]
    python -m pass_attention_gb300.profile_case decode [--B --H --Lmax --splits] [--reps N]
    python -m pass_attention_gb300.profile_case merge [--B --H --Lmax --splits] [--reps N]

``merge`` runs the split-KV decode once and then the merge ``--reps`` times on
its partials: the merge's inputs are the decode's (B, H, splits) partial
arrays, whose size does not depend on Lmax, so a short cache gives the same
merge launch with little memory held.

``--no-ws`` calls ``os_softmax_rows`` / ``os_softmax_rows_16bit`` without a
workspace, so rows over 1.6 MB take the kernels that stream them twice from
HBM instead of the cooperative one that re-reads them from L2.

Inputs are the seeded synthetic ones of ``workloads``; every call is
followed by a device synchronise, so a profiler filter such as
``-k regex:attn_fwd -s 1 -c 1`` captures one warm launch.
"""

from __future__ import annotations

import argparse
import ctypes
import math

import torch

import pass_attention_gb300 as oss
from pass_attention_gb300 import workloads


def _no_ws(x, y, kind):
    """One call of os_softmax_rows (kind None) or os_softmax_rows_16bit
    without a workspace."""
    rows, cols = x.shape
    m = torch.empty(rows, device=x.device)
    l = torch.empty(rows, device=x.device)
    lib = oss.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = (x.data_ptr(), y.data_ptr(), m.data_ptr(), l.data_ptr(), rows, cols, x.stride(0),
            y.stride(0), ctypes.c_float(1.0))
    if kind is None:
        st = lib.os_softmax_rows(*args, stream)
    else:
        st = lib.os_softmax_rows_16bit(*args, kind, stream)
    if st != 0:
        raise oss.OssError(st, "softmax without a workspace")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["softmax", "softmax16", "multipass", "attn", "decode", "merge"])
    ap.add_argument("--passes", type=int, default=3)
    ap.add_argument("--rows", type=int, default=32768)
    ap.add_argument("--cols", type=int, default=8192)
    ap.add_argument("--B", type=int, default=None)
    ap.add_argument("--H", type=int, default=None)
    ap.add_argument("--S", type=int, default=4096)
    ap.add_argument("--Lmax", type=int, default=32768)
    ap.add_argument("--splits", type=int, default=16)
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--dtype", choices=["bf16", "f16"], default="bf16")
    ap.add_argument("--no-ws", action="store_true")
    a = ap.parse_args(argv)
    oss.load()
    if a.case == "softmax":
        x = workloads.logits(a.rows, a.cols, 10.0, seed=1, device="cuda")
        y = torch.empty_like(x)
        for _ in range(a.reps):
            if a.no_ws:
                _no_ws(x, y, None)
            else:
                oss.softmax_rows(x, 1.0, y=y)
            torch.cuda.synchronize()
    elif a.case == "softmax16":
        dtype = torch.bfloat16 if a.dtype == "bf16" else torch.float16
        x = workloads.logits(a.rows, a.cols, 10.0, seed=1, device="cuda").to(dtype)
        y = torch.empty_like(x)
        for _ in range(a.reps):
            if a.no_ws:
                _no_ws(x, y, 2 if a.dtype == "f16" else 1)
            else:
                oss.softmax_rows_16bit(x, 1.0, y=y)
            torch.cuda.synchronize()
    elif a.case == "multipass":
        x = workloads.logits(a.rows, a.cols, 10.0, seed=1, device="cuda")
        y = torch.empty_like(x)
        for _ in range(a.reps):
            oss.softmax_rows_multipass(x, a.passes, 1.0, y=y)
            torch.cuda.synchronize()
    elif a.case == "attn":
        B, H = a.B or 4, a.H or 16
        q, k, v = workloads.qkv(B, H, a.S, a.S, 128, seed=2, device="cuda")
        for _ in range(a.reps):
            oss.attention_fwd(q, k, v, 1.0 / math.sqrt(128), a.causal)
            torch.cuda.synchronize()
        oss.check_device_error()
    elif a.case == "merge":
        B, H = a.B or 64, a.H or 32
        q, k, v, kv = workloads.decode_inputs(B, H, a.Lmax, 128, seed=4, device="cuda")
        pm, pl, po = oss.attention_decode_splitkv(q, k, v, kv, a.splits)
        del k, v
        torch.cuda.synchronize()
        o = torch.empty((B, H, 128), dtype=torch.bfloat16, device="cuda")
        for _ in range(a.reps):
            oss.merge_partials(pm, pl, po, finalize=True, o_out=o)
            torch.cuda.synchronize()
    else:
        B, H = a.B or 8, a.H or 32
        q, k, v, kv = workloads.decode_inputs(B, H, a.Lmax, 128, seed=4, device="cuda")
        for _ in range(a.reps):
            pm, pl, po = oss.attention_decode_splitkv(q, k, v, kv, a.splits)
            oss.merge_partials(pm, pl, po, finalize=True)
            torch.cuda.synchronize()
        print("kv_len sum", int(kv.sum().item()))
    print("done", a.case)


if __name__ == "__main__":
    main()
