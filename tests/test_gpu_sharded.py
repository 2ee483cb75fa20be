"""Sequence-sharded attention: per-shard partial states from
os_attention_fwd_partial, merged with os_merge_partials, equal the attention
over the whole sequence (the associative merge the curionode page names for
combining partial results across devices; here the shards run one after
another on one GPU) (GPU)."""

import math

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


def empty_partials(B, H, Sq, S, D=128):
    pm = torch.full((B, H, Sq, S), -math.inf, device="cuda")
    pl = torch.zeros((B, H, Sq, S), device="cuda")
    po = torch.zeros((B, H, Sq, S, D), device="cuda")
    return pm, pl, po


@pytest.mark.parametrize("bounds", [[0, 256, 700, 1000], [0, 1000], [0, 1, 129, 1000]])
def test_noncausal_shards_merge_to_full(bounds):
    B, H, Sq = 2, 2, 300
    Sk = bounds[-1]
    q, k, v = workloads.qkv(B, H, Sq, Sk, 128, seed=len(bounds) * 7 + Sk, device="cuda")
    scale = 1 / math.sqrt(128)
    n = len(bounds) - 1
    pm, pl, po = empty_partials(B, H, Sq, n)
    for s in range(n):
        lo, hi = bounds[s], bounds[s + 1]
        oss.attention_fwd_partial(q, k[:, :, lo:hi].contiguous(), v[:, :, lo:hi].contiguous(),
                                  pm, pl, po, s, scale)
    o, m, l, lse = oss.merge_partials(pm, pl, po, finalize=True)
    assert oss.check_device_error() == 0
    qh, kh, vh = f64(q), f64(k), f64(v)
    O, L = oracle.attention(qh, kh, vh, scale, False)
    A, _ = oracle.attention(qh, kh, np.abs(vh), scale, False)
    check_attn(f64(o), O, "merged O")
    check_attn(f64(lse), L, "merged lse")
    e_s = score_error_bound(qh, kh, scale)
    worst = {"lse": check_lse_tight(f64(lse), L, lse_bar(e_s), "merged lse"),
             "O": check_o_tight(f64(o), O, o_bar(O, A, e_s, Sk), "merged")}
    # each shard's partial state is the definition over that shard's keys
    pmh, plh, poh = f64(pm), f64(pl), f64(po)
    for s in range(n):
        lo, hi = bounds[s], bounds[s + 1]
        Os, Ls = oracle.attention(qh, kh[:, :, lo:hi], vh[:, :, lo:hi], scale, False)
        As, _ = oracle.attention(qh, kh[:, :, lo:hi], np.abs(vh[:, :, lo:hi]), scale, False)
        check_attn(pmh[..., s] + np.log(plh[..., s]), Ls, f"shard {s} lse")
        check_attn(poh[..., s, :] / plh[..., s, None], Os, f"shard {s} O/l")
        S = scale * np.einsum("bhqd,bhkd->bhqk", qh, kh[:, :, lo:hi])
        check_attn(pmh[..., s], S.max(axis=-1), f"shard {s} m")
        es = score_error_bound(qh, kh[:, :, lo:hi], scale)
        worst[f"shard{s} lse"] = check_lse_tight(pmh[..., s] + np.log(plh[..., s]), Ls, lse_bar(es),
                                                 f"shard {s} lse")
        worst[f"shard{s} m"] = check_lse_tight(pmh[..., s], S.max(axis=-1), lse_bar(es),
                                               f"shard {s} m")
        worst[f"shard{s} O"] = check_o_tight(poh[..., s, :] / plh[..., s, None], Os,
                                             o_bar(Os, As, es, hi - lo), f"shard {s}")
    report(f"shards {bounds}", **worst)


def test_causal_ring_assembly():
    # a causal sequence of 3 shards: query shard a takes full partials of key
    # shards b < a and a causal partial of its own shard
    B, H, S, n = 1, 2, 768, 3
    w = S // n
    q, k, v = workloads.qkv(B, H, S, S, 128, seed=33, device="cuda")
    scale = 1 / math.sqrt(128)
    qh, kh, vh = f64(q), f64(k), f64(v)
    O_ref, L_ref = oracle.attention(qh, kh, vh, scale, True)
    A_ref, _ = oracle.attention(qh, kh, np.abs(vh), scale, True)
    e_s = score_error_bound(qh, kh, scale)
    worst = {"lse": 0.0, "O": 0.0}
    for a in range(n):
        qa = q[:, :, a * w:(a + 1) * w].contiguous()
        pm, pl, po = empty_partials(B, H, w, n)
        for b in range(a + 1):
            kb = k[:, :, b * w:(b + 1) * w].contiguous()
            vb = v[:, :, b * w:(b + 1) * w].contiguous()
            oss.attention_fwd_partial(qa, kb, vb, pm, pl, po, b, scale, causal=(b == a))
        o, _, _, lse = oss.merge_partials(pm, pl, po, finalize=True)
        assert oss.check_device_error() == 0
        rows = slice(a * w, (a + 1) * w)
        check_attn(f64(o), O_ref[:, :, rows], f"query shard {a} O")
        check_attn(f64(lse), L_ref[:, :, rows], f"query shard {a} lse")
        worst["lse"] = max(worst["lse"], check_lse_tight(f64(lse), L_ref[:, :, rows],
                                                         lse_bar(e_s[:, :, rows]),
                                                         f"query shard {a} lse"))
        worst["O"] = max(worst["O"], check_o_tight(
            f64(o), O_ref[:, :, rows], o_bar(O_ref[:, :, rows], A_ref[:, :, rows],
                                             e_s[:, :, rows], S), f"query shard {a}"))
    report("causal ring", **worst)
