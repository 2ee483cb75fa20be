"""Seeded random shapes for every entry point, against the oracle (GPU).

The shape tests elsewhere pick their cases by hand (tile edges, ragged tails,
empty rows). Here one fixed seed draws the remaining combinations: row
counts, lengths that straddle the register/stream boundary, leading
dimensions, base offsets, scales, mask densities, KV lengths, split and shard
counts. Each case is a parametrised test whose id holds its draw, so a failure
names a case that can be re-run on its own."""

import math

import numpy as np
import pytest
import torch

import oracle
import pass_attention_gb300 as oss
from pass_attention_gb300 import workloads
from parity import check_attn, check_softmax, check_softmax16, f32

pytestmark = pytest.mark.gpu

_RNG = np.random.default_rng(20261202)


def _length(lo, hi):
    """Half the draws log-uniform (short lengths, tile edges), half uniform
    (the long lengths that run many tiles or leave the register path)."""
    if _RNG.integers(0, 2):
        return int(_RNG.integers(lo, hi + 1))
    return int(round(math.exp(_RNG.uniform(math.log(lo), math.log(hi)))))


def f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


# ---------------------------------------------------------------------------
# row softmax: fp32, 16-bit, the comparators
# ---------------------------------------------------------------------------

def _softmax_cases(n, elem_align):
    cases = []
    for _ in range(n):
        cols = _length(1, 70000)
        rows = int(_RNG.integers(1, max(2, min(64, 1_500_000 // cols)) + 1))
        layout = str(_RNG.choice(["aligned", "padded", "odd_ld", "offset"]))
        if layout == "aligned":
            ld = -(-cols // elem_align) * elem_align
        elif layout == "padded":
            ld = -(-cols // elem_align) * elem_align + elem_align * int(_RNG.integers(1, 5))
        elif layout == "odd_ld":
            ld = cols + int(_RNG.integers(0, elem_align))
        else:
            ld = cols
        scale = float(math.exp(_RNG.uniform(math.log(0.05), math.log(20.0))))
        mask = float(_RNG.choice([0.0, 0.0, 0.1, 0.9]))
        dead_row = bool(_RNG.integers(0, 4) == 0)
        cases.append((rows, cols, ld, layout, round(scale, 4), mask, dead_row))
    return cases


SOFTMAX_CASES = _softmax_cases(24, 4)
SOFTMAX16_CASES = [c + (str(_RNG.choice(["bf16", "f16"])),) for c in _softmax_cases(16, 8)]
MULTIPASS_CASES = [c + (int(_RNG.integers(2, 4)),) for c in _softmax_cases(8, 4)]


def _ids(cases):
    return ["-".join(str(v) for v in c) for c in cases]


def _input(rows, cols, ld, layout, mask, dead_row, seed, dtype):
    """x as a [rows, cols] view with row stride ld (offset by one element for
    the 'offset' layout), masked entries -inf, optionally one row all -inf."""
    if layout == "offset":
        buf = workloads.logits(1, rows * cols + 1, 10.0, seed, device="cuda").to(dtype)
        x = buf[0, 1:].view(rows, cols)
    else:
        x = workloads.logits(rows, ld, 10.0, seed, device="cuda").to(dtype)[:, :cols]
    if mask > 0.0:
        g = torch.Generator(device="cuda").manual_seed(seed + 1)
        x[torch.rand(x.shape, generator=g, device="cuda") < mask] = -float("inf")
    if dead_row:
        x[rows // 2] = -float("inf")
    return x


def _output_like(x, layout, ld):
    rows, cols = x.shape
    if layout == "offset":
        return torch.empty(rows * cols + 1, dtype=x.dtype, device="cuda")[1:].view(rows, cols)
    return torch.empty((rows, ld), dtype=x.dtype, device="cuda")[:, :cols]


@pytest.mark.parametrize("case", SOFTMAX_CASES, ids=_ids(SOFTMAX_CASES))
def test_softmax_rows_random(case):
    rows, cols, ld, layout, scale, mask, dead_row = case
    x = _input(rows, cols, ld, layout, mask, dead_row, rows * 7 + cols, torch.float32)
    y = _output_like(x, layout, ld)
    y, m, l = oss.softmax_rows(x, scale, y=y)
    torch.cuda.synchronize()
    check_softmax(y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                  *oracle.softmax_rows(x.cpu().numpy(), f32(scale)), what=str(case))


@pytest.mark.parametrize("case", SOFTMAX16_CASES, ids=_ids(SOFTMAX16_CASES))
def test_softmax_rows_16bit_random(case):
    rows, cols, ld, layout, scale, mask, dead_row, kind = case
    dtype = torch.bfloat16 if kind == "bf16" else torch.float16
    x = _input(rows, cols, ld, layout, mask, dead_row, rows * 11 + cols, dtype)
    y = _output_like(x, layout, ld)
    y, m, l = oss.softmax_rows_16bit(x, scale, y=y)
    torch.cuda.synchronize()
    xr = x.float().cpu().numpy().astype(np.float64)
    check_softmax16(y.float().cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                    *oracle.softmax_rows(xr, f32(scale)), kind=kind, what=str(case))


@pytest.mark.parametrize("case", MULTIPASS_CASES, ids=_ids(MULTIPASS_CASES))
def test_softmax_rows_multipass_random(case):
    rows, cols, ld, layout, scale, mask, dead_row, passes = case
    x = _input(rows, cols, ld, layout, mask, dead_row, rows * 13 + cols, torch.float32)
    y = _output_like(x, layout, ld)
    y, m, l = oss.softmax_rows_multipass(x, passes, scale, y=y)
    torch.cuda.synchronize()
    check_softmax(y.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(),
                  *oracle.softmax_rows(x.cpu().numpy(), f32(scale)), what=str(case))


# ---------------------------------------------------------------------------
# attention forward, sharded partials, split-KV decode, merge
# ---------------------------------------------------------------------------

def _attn_cases(n):
    cases = []
    while len(cases) < n:
        B, H = int(_RNG.integers(1, 3)), int(_RNG.integers(1, 4))
        causal = bool(_RNG.integers(0, 3) == 0)
        Sq = _length(1, 1500)
        Sk = Sq if causal else _length(1, 1500)
        if B * H * Sq * Sk > 6_000_000:     # keeps the fp64 oracle to seconds
            continue
        scale = round(float(math.exp(_RNG.uniform(math.log(0.02), math.log(0.3)))), 4)
        cases.append((B, H, Sq, Sk, causal, scale))
    return cases


def _shard_cases(n):
    cases = []
    for B, H, Sq, Sk, _, scale in _attn_cases(n):
        k = int(_RNG.integers(1, min(4, Sk) + 1))
        cuts = sorted(int(c) for c in _RNG.choice(np.arange(1, Sk), size=k - 1, replace=False)) \
            if k > 1 else []
        cases.append((B, H, Sq, Sk, scale, tuple([0] + cuts + [Sk])))
    return cases


def _decode_cases(n):
    cases = []
    for _ in range(n):
        B, H = int(_RNG.integers(1, 7)), int(_RNG.integers(1, 5))
        Lmax = _length(1, 6000)
        kv = tuple(int(v) for v in _RNG.integers(1, Lmax + 1, size=B))
        S = int(_RNG.integers(1, 65))
        cases.append((B, H, Lmax, S, kv))
    return cases


def _merge_cases(n):
    return [(int(_RNG.integers(1, 300)), int(_RNG.integers(1, 65)), 4 * int(_RNG.integers(1, 65)),
             round(float(_RNG.uniform(0.0, 0.6)), 2)) for _ in range(n)]


ATTN_CASES = _attn_cases(14)
SHARD_CASES = _shard_cases(6)
DECODE_CASES = _decode_cases(10)
MERGE_CASES = _merge_cases(10)


@pytest.mark.parametrize("case", ATTN_CASES, ids=_ids(ATTN_CASES))
def test_attention_fwd_random(case):
    B, H, Sq, Sk, causal, scale = case
    q, k, v = workloads.qkv(B, H, Sq, Sk, 128, seed=B * 7 + H * 131 + Sq * 17 + Sk, device="cuda")
    o, lse = oss.attention_fwd(q, k, v, scale, causal)
    assert oss.check_device_error() == 0
    O, L = oracle.attention(f64(q), f64(k), f64(v), f32(scale), causal)
    check_attn(f64(o), O, f"{case} O")
    check_attn(f64(lse), L, f"{case} lse")


@pytest.mark.parametrize("case", SHARD_CASES, ids=_ids(SHARD_CASES))
def test_sharded_partials_merge_random(case):
    B, H, Sq, Sk, scale, bounds = case
    q, k, v = workloads.qkv(B, H, Sq, Sk, 128, seed=Sq * 3 + Sk, device="cuda")
    n = len(bounds) - 1
    pm = torch.full((B, H, Sq, n), -math.inf, device="cuda")
    pl = torch.zeros((B, H, Sq, n), device="cuda")
    po = torch.zeros((B, H, Sq, n, 128), device="cuda")
    for s in range(n):
        lo, hi = bounds[s], bounds[s + 1]
        oss.attention_fwd_partial(q, k[:, :, lo:hi].contiguous(), v[:, :, lo:hi].contiguous(),
                                  pm, pl, po, s, scale)
    o, m, l, lse = oss.merge_partials(pm, pl, po, finalize=True)
    assert oss.check_device_error() == 0
    O, L = oracle.attention(f64(q), f64(k), f64(v), f32(scale), False)
    check_attn(f64(o), O, f"{case} merged O")
    check_attn(f64(lse), L, f"{case} merged lse")


@pytest.mark.parametrize("case", DECODE_CASES, ids=_ids(DECODE_CASES))
def test_decode_merge_random(case):
    B, H, Lmax, S, kv = case
    q, k, v, kvl = workloads.decode_inputs(B, H, Lmax, 128, seed=B + H * 10 + Lmax, device="cuda",
                                           kv_len=torch.tensor(kv))
    scale = 1.0 / math.sqrt(128)
    pm, pl, po = oss.attention_decode_splitkv(q, k, v, kvl, S, scale)
    o, m, l, lse = oss.merge_partials(pm, pl, po, finalize=True)
    torch.cuda.synchronize()
    qh, kh, vh = f64(q), f64(k), f64(v)
    O, L = oracle.decode(qh, kh, vh, list(kv), scale)
    check_attn(f64(o), O, f"{case} O")
    check_attn(f64(lse), L, f"{case} lse")
    # the partials themselves: empty splits exactly (-inf, 0, 0), the rest the
    # definition over the split's keys
    rm, rl, ro = oracle.decode_partials(qh, kh, vh, list(kv), S, scale)
    pmh, plh, poh = f64(pm), f64(pl), f64(po)
    empty = np.isneginf(rm)
    assert np.all(np.isneginf(pmh[empty])) and np.all(plh[empty] == 0.0)
    assert np.all(poh[empty] == 0.0)
    full = ~empty
    check_attn(pmh[full] + np.log(plh[full]), rm[full] + np.log(rl[full]), f"{case} part lse")
    check_attn(poh[full] / plh[full][:, None], ro[full] / rl[full][:, None], f"{case} part O/l")


@pytest.mark.parametrize("case", MERGE_CASES, ids=_ids(MERGE_CASES))
def test_merge_random(case):
    G, S, D, p_empty = case
    g = torch.Generator().manual_seed(G * 1000 + S * 10 + D)
    pm = torch.randn(G, S, generator=g, dtype=torch.float64) * 8
    pl = torch.rand(G, S, generator=g, dtype=torch.float64) * 99 + 1
    po = torch.randn(G, S, D, generator=g, dtype=torch.float64) * 10
    empty = torch.rand(G, S, generator=g) < p_empty
    pm[empty], pl[empty], po[empty] = -math.inf, 0.0, 0.0
    pm, pl, po = pm.float(), pl.float(), po.float()
    o, m, l, lse = oss.merge_partials(pm.cuda(), pl.cuda(), po.cuda(), finalize=True)
    On, rm, rl, rlse = oracle.merge(pm.double().numpy(), pl.double().numpy(), po.double().numpy())
    torch.cuda.synchronize()
    check_attn(f64(o), On, f"{case} O")
    check_attn(f64(lse), rlse, f"{case} lse")
    fin = np.isfinite(rm)
    assert np.all(np.isneginf(f64(m)[~fin])) and np.all(f64(l)[~fin] == 0.0)
    np.testing.assert_allclose(f64(m)[fin], rm[fin], rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(f64(l)[fin], rl[fin], rtol=1e-5)
