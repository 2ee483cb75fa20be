"""The seeded input recipe on CPU: each generator is deterministic per seed,
has the stated shape, type and distribution, and the named workloads carry
the sizes, seeds and options of the measured configurations."""

import math

import numpy as np
import torch

from pass_attention_gb300 import workloads as wl


def test_logits_are_seeded_normal_times_mult():
    a = wl.logits(300, 1000, 10.0, seed=7)
    b = wl.logits(300, 1000, 10.0, seed=7)
    c = wl.logits(300, 1000, 10.0, seed=8)
    assert a.dtype == torch.float32 and a.shape == (300, 1000)
    assert torch.equal(a, b) and not torch.equal(a, c)
    # the same draw without the multiplier, times 10, in fp32
    assert torch.equal(a, wl.logits(300, 1000, 1.0, seed=7) * 10.0)
    x = a.double().numpy() / 10.0
    n = x.size
    assert abs(x.mean()) < 5 / math.sqrt(n)
    assert abs(x.std() - 1.0) < 5 / math.sqrt(2 * n)
    assert abs(np.mean(np.abs(x) < 1.0) - 0.6827) < 0.005


def test_qkv_are_bf16_roundings_of_seeded_normals():
    q, k, v = wl.qkv(2, 3, 50, 70, 16, seed=5)
    assert q.shape == (2, 3, 50, 16) and k.shape == (2, 3, 70, 16) and v.shape == (2, 3, 70, 16)
    assert all(t.dtype == torch.bfloat16 for t in (q, k, v))
    g = torch.Generator().manual_seed(5)
    ref = [torch.randn((2, 3, S, 16), generator=g, dtype=torch.float32) for S in (50, 70, 70)]
    for t, r in zip((q, k, v), ref):
        assert torch.equal(t, r.to(torch.bfloat16))   # round to nearest even, once
    assert not torch.equal(k, v)
    q2, _, _ = wl.qkv(2, 3, 50, 70, 16, seed=5)
    assert torch.equal(q, q2)


def test_decode_lengths_and_shapes():
    q, k, v, kv = wl.decode_inputs(16, 2, 300, 8, seed=4)
    assert q.shape == (16, 2, 8) and k.shape == (16, 2, 300, 8) and v.shape == (16, 2, 300, 8)
    assert kv.dtype == torch.int32 and kv.shape == (16,)
    assert int(kv.min()) >= 1 and int(kv.max()) <= 300
    q2, k2, v2, kv2 = wl.decode_inputs(16, 2, 300, 8, seed=4)
    assert torch.equal(kv, kv2) and torch.equal(k, k2) and torch.equal(v, v2)
    _, _, _, given = wl.decode_inputs(3, 1, 40, 4, seed=1, kv_len=torch.tensor([40, 1, 17]))
    assert given.tolist() == [40, 1, 17] and given.dtype == torch.int32
    # lengths spread over the whole range
    _, _, _, many = wl.decode_inputs(512, 1, 1000, 1, seed=9)
    assert int(many.min()) < 50 and int(many.max()) > 950


def test_named_workloads():
    assert (wl.ROW64.rows, wl.ROW64.cols, wl.ROW64.mult, wl.ROW64.scale, wl.ROW64.seed) == (1, 64, 1.0, 1.0, 0)
    s = wl.SOFTMAX_32K
    assert (s.rows, s.cols, s.mult, s.scale, s.seed) == (32768, 8192, 10.0, 1.0, 1)
    a = wl.ATTN_4K
    assert (a.B, a.H, a.S, a.D, a.causal, a.seed) == (4, 16, 4096, 128, False, 2)
    c = wl.ATTN_CAUSAL
    assert (c.B, c.H, c.S, c.D, c.causal, c.seed) == (1, 32, 16384, 128, True, 3)
    d = wl.DECODE_64X32
    assert (d.B, d.H, d.D, d.Lmax, d.num_splits, d.seed) == (64, 32, 128, 32768, 16, 4)
    assert a.scale == 1.0 / math.sqrt(128) and d.scale == 1.0 / math.sqrt(128)
    assert set(wl.WORKLOADS) == {"row64", "softmax_32k", "attn_4k", "attn_causal", "decode_64x32"}
