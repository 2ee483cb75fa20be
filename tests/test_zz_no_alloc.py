"""os_attention_fwd_noalloc: the attention forward for callers that cannot
allocate device memory, such as a plugin that its host framework hands only
input and output buffers, or a latency-critical thread that must not call
cudaMalloc. It takes the split tail's workspace from a fixed array that the
library declares in device memory instead of one the caller allocates.

The GPU tests call it through the C ABI, twice in a row on each shape, and
compare both results with os_attention_fwd_ws (the binding's attention_fwd,
whose workspace the binding allocates) within the tolerance the split-tail
tests use, and with the oracle on sampled rows. This file is named to be
collected last, so that it also runs after every other test has used the
library; it passes alone in a fresh process as well."""

import ctypes
import math

import numpy as np
import pytest
import torch

import pass_attention_gb300 as oss
from pass_attention_gb300 import workloads


def noalloc(q, k, v, scale, causal=False):
    """One call of os_attention_fwd_noalloc on preallocated outputs."""
    B, H, Sq, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), device=q.device)
    st = oss.load().os_attention_fwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Sq,
        k.shape[2], D, ctypes.c_float(scale), int(causal),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, oss.load().os_status_string(st)
    return o, lse


def same_within_split_tolerance(o, lse, o_ref, lse_ref):
    """The bar the split-tail tests hold os_attention_fwd_ws to against the
    unsplit call: lse within 1e-4, O within bf16 rounding of its largest entry."""
    assert torch.allclose(lse, lse_ref, atol=1e-4, rtol=0)
    err = (o.float() - o_ref.float()).abs().max().item()
    assert err <= 2.0 ** -7 * (o_ref.float().abs().max().item() + 1e-3)


def test_noalloc_rejects_bad_arguments_without_a_gpu():
    # argument errors come back before anything touches a device
    lib = oss.load()
    p = ctypes.c_void_p(16)
    bad = [
        (0, 1, 128, 128, 128),    # B = 0
        (1, 1, 128, 128, 64),     # D other than 128
        (1, 1, -1, 128, 128),     # negative Sq
    ]
    for B, H, Sq, Sk, D in bad:
        st = lib.os_attention_fwd_noalloc(p, p, p, p, None, B, H, Sq, Sk, D,
                                          ctypes.c_float(1.0), 0, None)
        assert st != 0


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Sq,Sk", [
    (2, 3, 300, 200),     # 18 ragged query tiles, each cut in 2 parts
    (5, 16, 2000, 1000),  # 8 full rounds of the SMs, then 64 tiles in 2 parts
    (1, 1, 1024, 4096),   # 8 query tiles, each cut in 8 parts
])
def test_noalloc_matches_the_workspace_call_twice(B, H, Sq, Sk):
    from test_gpu_attention import check_rows

    scale = 1.0 / math.sqrt(128)
    q, k, v = workloads.qkv(B, H, Sq, Sk, 128, seed=B * 11 + Sq + Sk, device="cuda")
    assert oss.attention_fwd_workspace_bytes(B, H, Sq, Sk) > 0, "shape chosen to split"
    o_ref, lse_ref = oss.attention_fwd(q, k, v, scale)
    o1, lse1 = noalloc(q, k, v, scale)
    o2, lse2 = noalloc(q, k, v, scale)
    torch.cuda.synchronize()
    assert oss.check_device_error() == 0
    same_within_split_tolerance(o1, lse1, o_ref, lse_ref)
    same_within_split_tolerance(o2, lse2, o_ref, lse_ref)
    rng = np.random.default_rng(Sq + Sk)
    rows = list(zip(rng.integers(0, B, 256), rng.integers(0, H, 256), rng.integers(0, Sq, 256)))
    check_rows(q, k, v, o2, lse2, scale, False, rows, f"noalloc {B}x{H}x{Sq}x{Sk}")


@pytest.mark.gpu
def test_noalloc_shapes_in_a_row_share_the_array():
    # a shape with a wider split, then one with a narrower split, then one
    # with no split at all (causal): each call starts from the array as the
    # one before left it
    scale = 0.08
    cases = [(1, 1, 1024, 4096, False), (2, 3, 300, 200, False), (1, 2, 640, 640, True),
             (1, 1, 1024, 4096, False)]
    for B, H, Sq, Sk, causal in cases:
        q, k, v = workloads.qkv(B, H, Sq, Sk, 128, seed=Sq * 3 + Sk, device="cuda")
        o_ref, lse_ref = oss.attention_fwd(q, k, v, scale, causal=causal)
        o, lse = noalloc(q, k, v, scale, causal)
        torch.cuda.synchronize()
        assert oss.check_device_error() == 0
        same_within_split_tolerance(o, lse, o_ref, lse_ref)
