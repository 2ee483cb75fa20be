"""The secondary parity bars of tests/parity.py, checked on the CPU.

They must (1) admit what the kernels' arithmetic can legitimately produce
-- shown by evaluating the same definition with fp32 scores and sums and bf16
weights and outputs, the kernels' rounding points -- and (2) reject what a
scheduling or indexing bug produces at full size: the result with one KV tile
of 128 keys (attention) or one split of 16 (decode) left out, which the
spec bar (2e-2 + 2e-2 |ref|) still accepts. No kernel is involved: the
"broken" results are the oracle's own, over a reduced key set.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from pass_attention_gb300 import workloads
from parity import (check_attn, check_lse_tight, check_o_tight, lse_bar, o_bar,
                    score_error_bound)


def f64(t):
    return t.to(torch.float64).numpy()


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).to(
        torch.float64).numpy()


def emulate_rounding(q, k, v, scale):
    """The definition evaluated at the kernels' precisions: fp32 scores of
    exact products, fp32 weights and sum, weights rounded to bf16 for the
    weighted sum of V, O rounded to bf16. q [n, D], k, v [L, D]."""
    s = (q.astype(np.float32) @ k.astype(np.float32).T) * np.float32(scale)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m).astype(np.float32)
    l = p.sum(axis=1, dtype=np.float32)
    o = (bf16(p).astype(np.float32) @ v.astype(np.float32)) / l[:, None]
    lse = m[:, 0].astype(np.float64) + np.log(l.astype(np.float64))
    return bf16(o), lse


@pytest.fixture(scope="module")
def attn_rows():
    # 48 query rows against the 4096 keys of one attn_4k head
    w = workloads.ATTN_4K
    q, k, v = workloads.qkv(1, 1, 48, w.S, w.D, seed=w.seed)
    return f64(q)[0, 0], f64(k)[0, 0], f64(v)[0, 0], w.scale


def test_bars_admit_kernel_precision(attn_rows):
    q, k, v, scale = attn_rows
    O, L = oracle.attention(q[None, None], k[None, None], v[None, None], scale)
    A, _ = oracle.attention(q[None, None], k[None, None], np.abs(v)[None, None], scale)
    O, L, A = O[0, 0], L[0, 0], A[0, 0]
    o32, lse32 = emulate_rounding(q, k, v, scale)
    e_s = score_error_bound(q, k, scale)
    r_l = check_lse_tight(lse32, L, lse_bar(e_s), "emulated lse")
    r_o = check_o_tight(o32, O, o_bar(O, A, e_s, k.shape[0]), "emulated")
    assert r_l < 0.5 and r_o < 0.5


def test_dropped_kv_tile_fails_tight_bars_only(attn_rows):
    q, k, v, scale = attn_rows
    O, L = oracle.attention(q[None, None], k[None, None], v[None, None], scale)
    A, _ = oracle.attention(q[None, None], k[None, None], np.abs(v)[None, None], scale)
    O, L, A = O[0, 0], L[0, 0], A[0, 0]
    keep = np.ones(k.shape[0], dtype=bool)
    keep[1280:1408] = False   # one KV tile of 128 keys never visited
    Od, Ld = oracle.attention(q[None, None], k[keep][None, None], v[keep][None, None], scale)
    Od, Ld = Od[0, 0], Ld[0, 0]
    # the spec bar accepts the broken result ...
    check_attn(Od, O, "dropped tile O")
    check_attn(Ld, L, "dropped tile lse")
    # ... the secondary bars do not, on every row
    e_s = score_error_bound(q, k, scale)
    bar_l = lse_bar(e_s)
    assert np.all(np.abs(Ld - L) > 10 * bar_l)
    with pytest.raises(AssertionError):
        check_lse_tight(Ld, L, bar_l, "dropped tile lse")
    bar_o = o_bar(O, A, e_s, k.shape[0])
    assert np.mean(np.linalg.norm(Od - O, axis=1) > bar_o) > 0.9
    with pytest.raises(AssertionError):
        check_o_tight(Od, O, bar_o, "dropped tile")


def test_dropped_decode_split_fails_tight_bars_only():
    # one decode row of 32768 keys cut into 16 splits; merging 15 of them
    D, L, S = 128, 32768, 16
    q, k, v, _ = workloads.decode_inputs(1, 1, L, D, seed=4, kv_len=[L])
    qh, kh, vh = f64(q), f64(k), f64(v)
    scale = 1.0 / math.sqrt(D)
    pm, pl, po = oracle.decode_partials(qh, kh, vh, [L], S, scale)
    O_all, _, _, lse_all = oracle.merge(pm[0], pl[0], po[0])
    keep = [j for j in range(S) if j != 9]
    O_d, _, _, lse_d = oracle.merge(pm[0][:, keep], pl[0][:, keep], po[0][:, keep])
    check_attn(lse_d, lse_all, "dropped split lse")      # accepted by the spec bar
    check_attn(O_d, O_all, "dropped split O")
    e_s = score_error_bound(qh[0][:, None, :], kh[0], scale)[:, 0]
    with pytest.raises(AssertionError):
        check_lse_tight(lse_d, lse_all, lse_bar(e_s), "dropped split lse")


def test_score_bound_covers_fp32_scores(attn_rows):
    # the bound holds for fp32 scores summed in two different orders
    q, k, v, scale = attn_rows
    exact = scale * (q @ k.T)
    fwd = (q.astype(np.float32) @ k.astype(np.float32).T) * np.float32(scale)
    rev = (q[:, ::-1].astype(np.float32) @ k[:, ::-1].astype(np.float32).T) * np.float32(scale)
    e_s = score_error_bound(q, k, scale)
    for s in (fwd, rev):
        assert np.all(np.abs(s.astype(np.float64) - exact).max(axis=1) <= e_s)
