"""os_attention_fwd against the oracle's materialised attention (GPU)."""

import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import pass_attention_gb300 as oss
from pass_attention_gb300 import workloads
from parity import (check_attn, check_lse_tight, check_o_tight, lse_bar, o_bar, report,
                    score_error_bound)

pytestmark = pytest.mark.gpu


def f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def run(B, H, Sq, Sk, causal, seed, mult=1.0):
    q, k, v = workloads.qkv(B, H, Sq, Sk, 128, seed, device="cuda")
    if mult != 1.0:
        q = (q.float() * mult).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(128)
    o, lse = oss.attention_fwd(q, k, v, scale, causal)
    assert oss.check_device_error() == 0
    return q, k, v, o, lse, scale


def check_all_rows(q, k, v, o, lse, scale, causal, what, tight=True):
    """Every row against the oracle: the spec bar, and (tight) the
    secondary bars of tests/parity.py derived from the kernel's arithmetic."""
    qh, kh, vh = f64(q), f64(k), f64(v)
    B, H = q.shape[:2]
    Sk = k.shape[2]

    def one(bh):
        b, h = divmod(bh, H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        O, L = oracle.attention(qh[sl], kh[sl], vh[sl], scale, causal)
        A = oracle.attention(qh[sl], kh[sl], np.abs(vh[sl]), scale, causal)[0] if tight else None
        return bh, O[0, 0], L[0, 0], None if A is None else A[0, 0]

    on, ln = f64(o), f64(lse)
    worst = {"lse": 0.0, "O": 0.0}
    with ThreadPoolExecutor(max_workers=4) as ex:
        for bh, O, L, A in ex.map(one, range(B * H)):
            b, h = divmod(bh, H)
            check_attn(on[b, h], O, f"{what} O b{b} h{h}")
            check_attn(ln[b, h], L, f"{what} lse b{b} h{h}")
            if tight:
                e_s = score_error_bound(qh[b, h], kh[b, h], scale)
                worst["lse"] = max(worst["lse"], check_lse_tight(ln[b, h], L, lse_bar(e_s),
                                                                 f"{what} lse b{b} h{h}"))
                worst["O"] = max(worst["O"], check_o_tight(on[b, h], O, o_bar(O, A, e_s, Sk),
                                                           f"{what} b{b} h{h}"))
    if tight:
        report(what, **worst)


def check_rows(q, k, v, o, lse, scale, causal, rows, what):
    """Sampled rows (b, h, i) against the oracle, both bars."""
    qh, kh, vh = f64(q), f64(k), f64(v)
    O, L = oracle.attention(qh, kh, vh, scale, causal, rows=rows)
    A, _ = oracle.attention(qh, kh, np.abs(vh), scale, causal, rows=rows)
    on, ln = f64(o), f64(lse)
    got_o = np.stack([on[b, h, i] for b, h, i in rows])
    got_l = np.array([ln[b, h, i] for b, h, i in rows])
    check_attn(got_o, O, f"{what} O")
    check_attn(got_l, L, f"{what} lse")
    e_s = np.array([score_error_bound(qh[b, h, i][None], kh[b, h], scale)[0] for b, h, i in rows])
    r_l = check_lse_tight(got_l, L, lse_bar(e_s), f"{what} lse")
    r_o = check_o_tight(got_o, O, o_bar(O, A, e_s, k.shape[2]), what)
    report(what, lse=r_l, O=r_o)


@pytest.mark.parametrize("B,H,Sq,Sk", [
    (1, 1, 128, 128), (1, 2, 256, 256), (2, 3, 300, 200), (1, 1, 1, 1), (1, 1, 5, 700),
    (1, 2, 513, 1000), (2, 2, 1024, 384),
])
def test_noncausal_shapes(B, H, Sq, Sk):
    q, k, v, o, lse, scale = run(B, H, Sq, Sk, False, seed=Sq * 31 + Sk)
    check_all_rows(q, k, v, o, lse, scale, False, f"{B}x{H}x{Sq}x{Sk}")


@pytest.mark.parametrize("B,H,S", [(1, 1, 1), (1, 1, 129), (1, 2, 256), (1, 1, 300), (2, 2, 1000),
                                   (1, 2, 2048)])
def test_causal_shapes(B, H, S):
    q, k, v, o, lse, scale = run(B, H, S, S, True, seed=S * 17 + B)
    check_all_rows(q, k, v, o, lse, scale, True, f"causal {B}x{H}x{S}")


@pytest.mark.parametrize("B,H,Sq,Sk", [(3, 40, 300, 300), (2, 90, 130, 77)])
def test_noncausal_persistent_ragged_tiles(B, H, Sq, Sk):
    # more query tiles than SMs (360 and 360): each persistent CTA walks
    # several tiles, most with a ragged last query block and KV tile, so the
    # hand-over of Q, O and the step counters between tiles is exercised
    q, k, v, o, lse, scale = run(B, H, Sq, Sk, False, seed=B * 1000 + H + Sk)
    check_all_rows(q, k, v, o, lse, scale, False, f"persistent {B}x{H}x{Sq}x{Sk}")


def test_causal_first_row_is_first_value_and_zero_query_is_mean():
    q, k, v = workloads.qkv(1, 2, 700, 700, 128, seed=3, device="cuda")
    o, lse = oss.attention_fwd(q, k, v, 0.1, causal=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(f64(o)[:, :, 0], f64(v)[:, :, 0])  # bf16 round trip is exact
    z = torch.zeros_like(q)
    o, lse = oss.attention_fwd(z, k, v, 0.1, causal=False)
    torch.cuda.synchronize()
    mean = f64(v).mean(axis=2)
    check_attn(f64(o), np.broadcast_to(mean[:, :, None, :], o.shape), "mean of V")
    check_attn(f64(lse), np.full(lse.shape, math.log(700)), "lse uniform")


def test_large_logits_stay_finite():
    # |q.k| * scale in the hundreds: exponentials are only ever taken of
    # non-positive differences, so nothing overflows
    q, k, v, o, lse, scale = run(1, 2, 384, 640, False, seed=8, mult=30.0)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    check_all_rows(q, k, v, o, lse, scale, False, "x30")


@pytest.mark.parametrize("causal", [False, True])
def test_max_rising_every_tile(causal):
    # key norms grow along the sequence, so each 128-key tile raises every
    # row's maximum by far more than the 2^8 slack: the reference maximum and
    # the output accumulator are rescaled on every tile
    B, H, S = 1, 2, 1536
    q, k, v = workloads.qkv(B, H, S, S, 128, seed=12, device="cuda")
    grow = (1.0 + torch.arange(S, device="cuda", dtype=torch.float32) / 24.0)[None, None, :, None]
    k = (k.float() * grow).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(128)
    o, lse = oss.attention_fwd(q, k, v, scale, causal)
    assert oss.check_device_error() == 0
    check_all_rows(q, k, v, o, lse, scale, causal, "rising max")


def test_repeat_calls_identical():
    q, k, v = workloads.qkv(2, 2, 512, 512, 128, seed=4, device="cuda")
    o1, l1 = oss.attention_fwd(q, k, v, 0.1, causal=True)
    o2, l2 = oss.attention_fwd(q, k, v, 0.1, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.slow
def test_full_size_attn_4k_every_row():
    w = workloads.ATTN_4K
    q, k, v = workloads.qkv(w.B, w.H, w.S, w.S, w.D, w.seed, device="cuda")
    o, lse = oss.attention_fwd(q, k, v, w.scale, w.causal)
    assert oss.check_device_error() == 0
    check_all_rows(q, k, v, o, lse, w.scale, w.causal, "attn_4k")


@pytest.mark.slow
def test_full_size_attn_causal_sampled_rows():
    w = workloads.ATTN_CAUSAL
    q, k, v = workloads.qkv(w.B, w.H, w.S, w.S, w.D, w.seed, device="cuda")
    o, lse = oss.attention_fwd(q, k, v, w.scale, w.causal)
    assert oss.check_device_error() == 0
    rng = np.random.default_rng(w.seed)
    n = 4096
    rows = list(zip(rng.integers(0, w.B, n), rng.integers(0, w.H, n), rng.integers(0, w.S, n)))
    rows += [(0, h, i) for h in (0, w.H - 1) for i in (0, 1, 127, 128, 255, 256, w.S - 1)]
    check_rows(q, k, v, o, lse, w.scale, True, rows, "attn_causal")


def test_causal_beyond_the_schedule_size():
    # 8 x 950 heads of 128 queries: 2 causal query tiles per head, 15200 tiles,
    # more than the host-built schedule holds, so this launch takes one CTA per
    # tile; the other causal tests run on the schedule
    B, H, S = 8, 950, 128
    q, k, v = workloads.qkv(B, H, S, S, 128, seed=29, device="cuda")
    scale = 1.0 / math.sqrt(128)
    o, lse = oss.attention_fwd(q, k, v, scale, True)
    assert oss.check_device_error() == 0
    rng = np.random.default_rng(29)
    n = 2048
    rows = list(zip(rng.integers(0, B, n), rng.integers(0, H, n), rng.integers(0, S, n)))
    rows += [(b, h, i) for b, h in ((0, 0), (B - 1, H - 1)) for i in (0, 63, 64, 127)]
    check_rows(q, k, v, o, lse, scale, True, rows, "15200 tiles")


@pytest.mark.parametrize("policy", ["threshold", "on_rise", "always"])
@pytest.mark.parametrize("B,H,Sq,Sk,causal", [(2, 2, 1000, 700, False), (1, 2, 1000, 1000, True),
                                               (3, 40, 300, 300, False), (2, 3, 1, 129, False)])
def test_rescale_policies(policy, B, H, Sq, Sk, causal):
    # the three rescale policies compute the same result within the bars
    oss.set_rescale_policy(policy)
    try:
        assert oss.rescale_policy() == policy
        q, k, v, o, lse, scale = run(B, H, Sq, Sk, causal, seed=Sq + Sk + B)
    finally:
        oss.set_rescale_policy("threshold")
    check_all_rows(q, k, v, o, lse, scale, causal, f"{policy} {B}x{H}x{Sq}x{Sk}")


@pytest.mark.parametrize("policy", ["on_rise", "always"])
@pytest.mark.parametrize("causal", [False, True])
def test_rescale_policies_rising_max(policy, causal):
    # every tile raises every row's maximum: all policies rescale O each tile
    B, H, S = 1, 2, 1536
    q, k, v = workloads.qkv(B, H, S, S, 128, seed=12, device="cuda")
    grow = (1.0 + torch.arange(S, device="cuda", dtype=torch.float32) / 24.0)[None, None, :, None]
    k = (k.float() * grow).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(128)
    oss.set_rescale_policy(policy)
    try:
        o, lse = oss.attention_fwd(q, k, v, scale, causal)
        assert oss.check_device_error() == 0
    finally:
        oss.set_rescale_policy("threshold")
    check_all_rows(q, k, v, o, lse, scale, causal, f"{policy} rising max")


def test_rescale_policy_is_per_thread():
    import threading
    oss.set_rescale_policy("always")
    seen = []
    t = threading.Thread(target=lambda: seen.append(oss.rescale_policy()))
    t.start()
    t.join()
    oss.set_rescale_policy("threshold")
    assert seen == ["threshold"]


def _attn_no_split(q, k, v, scale):
    """os_attention_fwd without a workspace (whole query tiles only)."""
    import ctypes
    B, H, Sq, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), device=q.device)
    st = oss.load().os_attention_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), B, H, Sq, k.shape[2], D, ctypes.c_float(scale),
                                     0, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    return o, lse


@pytest.mark.parametrize("B,H,Sq,Sk", [
    (1, 1, 1024, 4096),   # 8 query tiles: each cut into 8 parts of 4 KV tiles
    (1, 2, 256, 129),     # 2 KV tiles, one key in the second: parts of one tile
    (2, 3, 300, 200),     # 18 ragged query tiles, 2 parts each
    (5, 16, 2000, 1000),  # 1280 tiles: 8 full rounds, then 64 tiles in 2 parts
    (4, 16, 4096, 640),   # the attn_4k tile count with fewer keys: 72 tiles split in 2
])
def test_split_tail_matches_oracle_and_unsplit(B, H, Sq, Sk):
    scale = 1.0 / math.sqrt(128)
    q, k, v = workloads.qkv(B, H, Sq, Sk, 128, seed=B * 7 + Sq + Sk, device="cuda")
    need = oss.attention_fwd_workspace_bytes(B, H, Sq, Sk)
    assert need > 0, "this shape was chosen to take the split tail"
    o, lse = oss.attention_fwd(q, k, v, scale)          # with the workspace
    o1, lse1 = _attn_no_split(q, k, v, scale)
    assert oss.check_device_error() == 0
    # the split result differs from the unsplit one only by the rounding of
    # the merge: lse within the tight bar of both, O within bf16 rounding
    assert torch.allclose(lse, lse1, atol=1e-4, rtol=0)
    assert (o.float() - o1.float()).abs().max().item() <= 2.0 ** -7 * (o1.float().abs().max().item() + 1e-3)
    if B * H * Sq <= 4096:
        check_all_rows(q, k, v, o, lse, scale, False, f"split {B}x{H}x{Sq}x{Sk}")
    else:
        rng = np.random.default_rng(Sq)
        rows = list(zip(rng.integers(0, B, 2048), rng.integers(0, H, 2048), rng.integers(0, Sq, 2048)))
        check_rows(q, k, v, o, lse, scale, False, rows, f"split {B}x{H}x{Sq}x{Sk}")
    # every completed call leaves the workspace's counters at zero
    sp = torch.cuda.current_stream().cuda_stream
    ws = oss._WORKSPACES[(q.device.index, sp, "attn")]
    torch.cuda.synchronize()
    tiles = B * H * ((Sq + 127) // 128)
    sms = torch.cuda.get_device_properties(q.device).multi_processor_count
    tail = tiles - (tiles // sms) * sms
    cnt = ws[need - tail * 8 * 4:need].view(torch.int32)
    assert int(cnt.abs().sum().item()) == 0


def test_split_tail_repeat_calls_identical():
    # the merge runs over the parts in part order, whichever SM merges
    q, k, v = workloads.qkv(2, 3, 640, 1500, 128, seed=21, device="cuda")
    assert oss.attention_fwd_workspace_bytes(2, 3, 640, 1500) > 0
    o1, l1 = oss.attention_fwd(q, k, v, 0.1)
    o2, l2 = oss.attention_fwd(q, k, v, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_no_workspace_for_causal_or_full_rounds():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert oss.attention_fwd_workspace_bytes(1, 32, 16384, 16384, causal=True) == 0
    # tiles that fill whole rounds: sms query tiles of 128 rows
    assert oss.attention_fwd_workspace_bytes(1, sms, 128, 4096) == 0


def test_split_tail_on_two_streams_keeps_workspaces_apart():
    # two launches that both take the split tail, on two streams with no
    # ordering between them: each stream gets its own workspace (counters and
    # partial states), and each result equals the same call made alone
    B, H, Sq, Sk = 2, 3, 640, 1500
    assert oss.attention_fwd_workspace_bytes(B, H, Sq, Sk) > 0
    q1, k1, v1 = workloads.qkv(B, H, Sq, Sk, 128, seed=31, device="cuda")
    q2, k2, v2 = workloads.qkv(B, H, Sq, Sk, 128, seed=32, device="cuda")
    ref1 = oss.attention_fwd(q1, k1, v1, 0.1)
    ref2 = oss.attention_fwd(q2, k2, v2, 0.1)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        with torch.cuda.stream(s1):
            o1, l1 = oss.attention_fwd(q1, k1, v1, 0.1, stream=s1)
        with torch.cuda.stream(s2):
            o2, l2 = oss.attention_fwd(q2, k2, v2, 0.1, stream=s2)
    torch.cuda.synchronize()
    assert oss.check_device_error() == 0
    assert torch.equal(o1, ref1[0]) and torch.equal(l1, ref1[1])
    assert torch.equal(o2, ref2[0]) and torch.equal(l2, ref2[1])
    dev = q1.device.index
    keys = {key for key in oss._WORKSPACES if key[0] == dev and key[2] == "attn"}
    assert (dev, s1.cuda_stream, "attn") in keys and (dev, s2.cuda_stream, "attn") in keys
