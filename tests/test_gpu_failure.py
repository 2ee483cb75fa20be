"""Failure detection without a GPU fault: a bounded wait inside the
attention kernel (one V tile is never loaded) or inside the cluster-resident
row softmax (a copy barrier expects 16 bytes that never come) is made to run
out, and the host reads the timeout through os_check_device_error. No trap,
no bad address, no endless wait; the context must stay usable (GPU)."""

import math

import numpy as np
import pytest
import torch

import oracle
import pass_attention_gb300 as oss
from pass_attention_gb300 import workloads
from parity import check_attn

pytestmark = pytest.mark.gpu

OS_ERR_TIMEOUT = 5
KERNEL_ATTN = 1
SITE_V_FULL = 3
SITE_O_DONE = 8


def f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def test_skipped_load_times_out_and_context_survives():
    # one 128-row query tile per SM (whole rounds: no split tail), four KV steps
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    q, k, v = workloads.qkv(1, sms, 128, 512, 128, seed=21, device="cuda")
    assert oss.attention_fwd_workspace_bytes(1, sms, 128, 512) == 0
    assert oss.check_device_error() == 0
    oss.debug_inject_fault(1, step=1, timeout_ns=20_000_000)  # 20 ms
    oss.attention_fwd(q, k, v, 1 / math.sqrt(128), False)
    with pytest.raises(oss.OssError) as info:
        oss.check_device_error()
    assert info.value.status == OS_ERR_TIMEOUT
    code = int(str(info.value).split("code ")[1].split(")")[0], 16)
    assert code & 0xFF == KERNEL_ATTN
    assert (code >> 8) & 0xFF == SITE_V_FULL
    # the word was cleared, and the same context computes correctly again
    assert oss.check_device_error() == 0
    o, lse = oss.attention_fwd(q, k, v, 1 / math.sqrt(128), False)
    assert oss.check_device_error() == 0
    O, L = oracle.attention(f64(q), f64(k), f64(v), 1 / math.sqrt(128), False)
    check_attn(f64(o), O, "after timeout O")
    check_attn(f64(lse), L, "after timeout lse")


def test_split_tail_part_times_out_and_context_survives():
    # 6 query tiles cut into 4 parts of one KV tile each: every part skips its
    # only V load; no part finishes, so no counter moves, and the next call on
    # the same workspace computes correctly
    q, k, v = workloads.qkv(1, 2, 384, 512, 128, seed=24, device="cuda")
    assert oss.attention_fwd_workspace_bytes(1, 2, 384, 512) > 0
    assert oss.check_device_error() == 0
    oss.debug_inject_fault(1, step=0, timeout_ns=20_000_000)
    oss.attention_fwd(q, k, v, 1 / math.sqrt(128), False)
    code = timeout_code()
    assert code & 0xFF == KERNEL_ATTN and (code >> 8) & 0xFF == SITE_V_FULL
    o, lse = oss.attention_fwd(q, k, v, 1 / math.sqrt(128), False)
    assert oss.check_device_error() == 0
    O, L = oracle.attention(f64(q), f64(k), f64(v), 1 / math.sqrt(128), False)
    check_attn(f64(o), O, "after split timeout O")
    check_attn(f64(lse), L, "after split timeout lse")


def test_fault_is_consumed_by_one_call():
    q, k, v = workloads.qkv(1, 1, 128, 256, 128, seed=22, device="cuda")
    oss.debug_inject_fault(1, step=0, timeout_ns=20_000_000)
    oss.debug_inject_fault(0)  # disarmed again
    oss.attention_fwd(q, k, v)
    assert oss.check_device_error() == 0


def test_timeout_stops_the_whole_launch():
    # a causal launch with more query tiles than the host-built schedule holds
    # (8 x 950 heads x 3 tiles = 22800) runs one CTA per tile, ~150 waves of
    # CTAs on 152 SMs; every CTA skips the V tile of its second KV step. The
    # first timeout is recorded with the launch's tag and the remaining CTAs
    # give up on their next poll, so the launch ends after about one timeout
    # (20 ms), not one per wave
    import time
    q, k, v = workloads.qkv(8, 950, 256, 256, 128, seed=23, device="cuda")
    assert oss.check_device_error() == 0
    torch.cuda.synchronize()
    oss.debug_inject_fault(1, step=1, timeout_ns=20_000_000)
    t0 = time.perf_counter()
    oss.attention_fwd(q, k, v, 1 / math.sqrt(128), True)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    with pytest.raises(oss.OssError) as info:
        oss.check_device_error()
    code = int(str(info.value).split("code ")[1].split(")")[0], 16)
    assert code & 0xFF == KERNEL_ATTN
    # the first wait to run out is recorded: the P V thread's on the missing
    # V tile, or, in another of the ~150 waves of CTAs, an epilogue's on that
    # P V (both follow from the same skipped load)
    assert (code >> 8) & 0xFF in (SITE_V_FULL, SITE_O_DONE)
    assert 1 <= (code >> 16) <= 65535  # the launch tag
    assert elapsed < 0.3, f"launch took {elapsed:.3f} s after the first timeout"
    # the context still works
    o, _ = oss.attention_fwd(q[:, :1, :256].contiguous(), k[:, :1, :256].contiguous(),
                             v[:, :1, :256].contiguous(), 1 / math.sqrt(128), True)
    assert oss.check_device_error() == 0


KERNEL_SOFTMAX_ROWS = 2
SITE_COPIES = 1
SITE_STATES = 2


def timeout_code():
    with pytest.raises(oss.OssError) as info:
        oss.check_device_error()
    assert info.value.status == OS_ERR_TIMEOUT
    return int(str(info.value).split("code ")[1].split(")")[0], 16)


@pytest.mark.parametrize("kind,cols,rows,site", [
    ("fp32", 65536, 200, SITE_STATES),   # 256 KB rows in the registers of a cluster of 8
    ("bf16", 131072, 64, SITE_STATES),   # the same, 16-bit
    ("bf16", 20000, 700, SITE_STATES),   # 40 KB rows in the registers of a cluster of 2
    ("fp32", 100000, 60, SITE_COPIES),   # 400 KB rows in a cluster's shared memory
    ("bf16", 20001, 700, SITE_COPIES),   # off the 16-byte grid, 40 KB: one CTA, two buffers
    ("bf16", 100, 100000, SITE_COPIES),  # 200-byte rows of a dense matrix: tiles staged
])
def test_row_softmax_wait_times_out_and_context_survives(kind, cols, rows, site):
    # every CTA's first row (or tile) expects 16 bytes that never arrive,
    # on its copies' barrier or on the barrier of the cluster's states: its
    # wait gives up after 20 ms, it waits (and copies or sends) no more, so
    # a peer waiting for it gives up too; every CTA still meets its barriers
    # and the launch ends
    import time
    dtype = torch.float32 if kind == "fp32" else torch.bfloat16
    x = workloads.logits(rows, cols, 10.0, seed=cols, device="cuda").to(dtype)
    call = oss.softmax_rows if kind == "fp32" else oss.softmax_rows_16bit
    call(x, 1.0)
    assert oss.check_device_error() == 0
    oss.debug_inject_fault(2, timeout_ns=20_000_000)
    t0 = time.perf_counter()
    call(x, 1.0)
    code = timeout_code()
    assert time.perf_counter() - t0 < 1.0
    assert code & 0xFF == KERNEL_SOFTMAX_ROWS
    assert (code >> 8) & 0xFF == site
    # the word was cleared, the hook consumed, and the context computes correctly
    assert oss.check_device_error() == 0
    y, m, l = call(x, 1.0)
    assert oss.check_device_error() == 0
    xr = x.float().cpu().numpy().astype(np.float64)
    ry, rm, rl = oracle.softmax_rows(xr, 1.0)
    assert np.array_equal(m.cpu().numpy(), rm.astype(np.float32))
    bar = 1e-5 if kind == "fp32" else 2.0 ** -8 + 1e-5
    assert np.all(np.abs(y.float().cpu().numpy() - ry) <= bar * ry + 2.0 ** -126)


def test_row_softmax_hook_ignored_off_the_cluster_path():
    # rows short enough for registers never wait on copies: the armed hook is
    # consumed without effect
    x = workloads.logits(64, 4096, 10.0, seed=3, device="cuda")
    oss.debug_inject_fault(2, timeout_ns=20_000_000)
    oss.softmax_rows(x, 1.0)
    assert oss.check_device_error() == 0
    oss.softmax_rows(workloads.logits(8, 100000, 10.0, seed=4, device="cuda"), 1.0)
    assert oss.check_device_error() == 0
