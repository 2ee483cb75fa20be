"""Failure detection without a GPU fault: a bounded wait inside the
attention kernel is made to run out (one V tile is never loaded), and the
host reads the timeout through os_check_device_error. No trap, no bad
address, no endless wait; the context must stay usable (GPU)."""

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


def f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def test_skipped_load_times_out_and_context_survives():
    q, k, v = workloads.qkv(1, 2, 384, 512, 128, seed=21, device="cuda")
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
    assert (code >> 8) & 0xFF == SITE_V_FULL
    assert 1 <= (code >> 16) <= 65535  # the launch tag
    assert elapsed < 0.3, f"launch took {elapsed:.3f} s after the first timeout"
    # the context still works
    o, _ = oss.attention_fwd(q[:, :1, :256].contiguous(), k[:, :1, :256].contiguous(),
                             v[:, :1, :256].contiguous(), 1 / math.sqrt(128), True)
    assert oss.check_device_error() == 0
