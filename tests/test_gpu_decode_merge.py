"""os_attention_decode_splitkv and os_merge_partials against the oracle (GPU)."""

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


def check_partials(pm, pl, po, rm, rl, ro, what, e_s=None, ra=None, Lk=None):
    """Compare partials by what they determine: m, lse = m + ln l and O / l;
    empty splits must be exactly (-inf, 0, 0). With e_s (the score error
    bound per (b, h)), ra (the oracle's partials of |V|) and Lk (keys per
    batch), also the secondary bars. Returns the largest ratios to those."""
    empty = np.isneginf(rm)
    assert np.all(np.isneginf(pm[empty])) and np.all(pl[empty] == 0.0), f"{what}: empty splits"
    assert np.all(po[empty] == 0.0), f"{what}: empty split O"
    full = ~empty
    assert np.all(np.isfinite(pm[full])) and np.all(pl[full] > 0), f"{what}: non-empty splits"
    check_attn(pm[full], rm[full], what + " part m")
    check_attn(pm[full] + np.log(pl[full]), rm[full] + np.log(rl[full]), what + " part lse")
    check_attn(po[full] / pl[full][:, None], ro[full] / rl[full][:, None], what + " part O/l")
    if e_s is None:
        return {}
    es = np.broadcast_to(np.asarray(e_s)[..., None], rm.shape)[full]
    bar = lse_bar(es)
    r_m = check_lse_tight(pm[full], rm[full], bar, what + " part m")
    r_l = check_lse_tight(pm[full] + np.log(pl[full]), rm[full] + np.log(rl[full]), bar,
                          what + " part lse")
    ref_o = ro[full] / rl[full][:, None]
    a_abs = ra[full] / rl[full][:, None]
    n = np.broadcast_to(np.asarray(Lk, dtype=np.float64).reshape(-1, 1, 1), rm.shape)[full]
    r_o = check_o_tight(po[full] / pl[full][:, None], ref_o, o_bar(ref_o, a_abs, es, n),
                        what + " part O/l")
    return {"part_m": r_m, "part_lse": r_l, "part_O": r_o}


def tight_merged(o, lse, qh, kh, vh, kvh, scale, what):
    """The merged output and lse against the oracle under the secondary bars."""
    O_ref, lse_ref = oracle.decode(qh, kh, vh, kvh, scale)
    A, _ = oracle.decode(qh, kh, np.abs(vh), kvh, scale)
    e_s = np.stack([score_error_bound(qh[b][:, None, :], kh[b, :, :int(kvh[b])], scale)[:, 0]
                    for b in range(qh.shape[0])])
    n = np.asarray(kvh, dtype=np.float64)[:, None]
    r_l = check_lse_tight(lse, lse_ref, lse_bar(e_s), what + " lse")
    r_o = check_o_tight(o, O_ref, o_bar(O_ref, A, e_s, n), what)
    return e_s, {"lse": r_l, "O": r_o}


def run_decode(B, H, Lmax, S, seed, kv_len=None):
    D = 128
    q, k, v, kv = workloads.decode_inputs(B, H, Lmax, D, seed, device="cuda", kv_len=kv_len)
    scale = 1.0 / math.sqrt(D)
    pm, pl, po = oss.attention_decode_splitkv(q, k, v, kv, S, scale)
    o, m, l, lse = oss.merge_partials(pm, pl, po, finalize=True)
    torch.cuda.synchronize()
    qh, kh, vh, kvh = f64(q), f64(k), f64(v), kv.cpu().numpy()
    what = f"decode {B}x{H}x{Lmax}/{S}"
    O_ref, lse_ref = oracle.decode(qh, kh, vh, kvh, scale)
    check_attn(f64(o), O_ref, "decode O")
    check_attn(f64(lse), lse_ref, "decode lse")
    e_s, worst = tight_merged(f64(o), f64(lse), qh, kh, vh, kvh, scale, what)
    rm, rl, ro = oracle.decode_partials(qh, kh, vh, kvh, S, scale)
    ra = oracle.decode_partials(qh, kh, np.abs(vh), kvh, S, scale)[2]
    worst.update(check_partials(f64(pm), f64(pl), f64(po), rm, rl, ro, what, e_s, ra, kvh))
    report(what, **worst)


@pytest.mark.parametrize("B,H,Lmax,S,kv_len", [
    (3, 4, 300, 16, [300, 5, 77]),      # ragged; 5 < 16 leaves splits empty
    (2, 3, 1, 16, [1, 1]),              # one key: O = v_0
    (2, 2, 1000, 1, [1000, 999]),       # no split at all
    (1, 2, 4099, 64, [4099]),           # most splits allowed, ragged tail
    (4, 2, 513, 7, [513, 1, 8, 64]),    # split count that does not divide
])
def test_decode_small(B, H, Lmax, S, kv_len):
    run_decode(B, H, Lmax, S, seed=B * 100 + S, kv_len=torch.tensor(kv_len))


def test_decode_random_lengths():
    run_decode(8, 8, 2048, 16, seed=44)


@pytest.mark.slow
def test_full_size_decode_every_row():
    # all B x H = 2048 query rows of the decode workload: each batch's keys
    # and values (up to 32768 x 32 heads) go to the host once, and the oracle
    # evaluates the partials of every split and the unsplit result for all of
    # that batch's heads
    w = workloads.DECODE_64X32
    q, k, v, kv = workloads.decode_inputs(w.B, w.H, w.Lmax, w.D, w.seed, device="cuda")
    pm, pl, po = oss.attention_decode_splitkv(q, k, v, kv, w.num_splits, w.scale)
    o, m, l, lse = oss.merge_partials(pm, pl, po, finalize=True)
    torch.cuda.synchronize()
    kvh = kv.cpu().numpy()
    qh, pmh, plh, poh, oh, lseh = f64(q), f64(pm), f64(pl), f64(po), f64(o), f64(lse)

    def one(item):
        b, kb, vb = item
        L = int(kvh[b])
        kb, vb = kb.to(torch.float64).numpy(), vb.to(torch.float64).numpy()
        rm, rl, ro = oracle.decode_partials(qh[b:b + 1], kb, vb, [L], w.num_splits, w.scale)
        ra = oracle.decode_partials(qh[b:b + 1], kb, np.abs(vb), [L], w.num_splits, w.scale)[2]
        O_ref, lse_ref = oracle.decode(qh[b:b + 1], kb, vb, [L], w.scale)
        e_s, r = tight_merged(oh[b:b + 1], lseh[b:b + 1], qh[b:b + 1], kb, vb, [L], w.scale,
                              f"decode b{b}")
        return b, rm, rl, ro, ra, O_ref, lse_ref, e_s, r

    worst = {}
    group = 8  # batches whose keys and values are on the host at once (<= ~2 GB of bf16)
    with ThreadPoolExecutor(max_workers=4) as ex:
        for b0 in range(0, w.B, group):
            # device-to-host copies on this thread (the only CUDA user)
            items = [(b, k[b:b + 1, :, :int(kvh[b])].cpu(), v[b:b + 1, :, :int(kvh[b])].cpu())
                     for b in range(b0, min(w.B, b0 + group))]
            for b, rm, rl, ro, ra, O_ref, lse_ref, e_s, r in ex.map(one, items):
                r.update(check_partials(pmh[b:b + 1], plh[b:b + 1], poh[b:b + 1], rm, rl, ro,
                                        f"decode b{b}", e_s, ra, [int(kvh[b])]))
                check_attn(oh[b:b + 1], O_ref, f"O b{b}")
                check_attn(lseh[b:b + 1], lse_ref, f"lse b{b}")
                for key, val in r.items():
                    worst[key] = max(worst.get(key, 0.0), val)
            del items
    report("decode_64x32", **worst)


# ---------------------------------------------------------------------------
# merge on its own
# ---------------------------------------------------------------------------

def random_partials(G, S, D, seed):
    g = torch.Generator().manual_seed(seed)
    pm = torch.randn(G, S, generator=g, dtype=torch.float64) * 5
    pl = torch.rand(G, S, generator=g, dtype=torch.float64) * 49 + 1
    po = torch.randn(G, S, D, generator=g, dtype=torch.float64) * 10
    empty = torch.rand(G, S, generator=g) < 0.25
    pm[empty] = -math.inf
    pl[empty] = 0.0
    po[empty] = 0.0
    pm[0] = -math.inf      # an all-empty group
    pl[0] = 0.0
    po[0] = 0.0
    return pm.float(), pl.float(), po.float()


@pytest.mark.parametrize("S", [1, 2, 5, 7, 16, 64])
@pytest.mark.parametrize("D", [4, 64, 128, 256])
def test_merge_finalize(S, D):
    pm, pl, po = random_partials(33, S, D, seed=S * 1000 + D)
    o, m, l, lse = oss.merge_partials(pm.cuda(), pl.cuda(), po.cuda(), finalize=True)
    On, rm, rl, rlse = oracle.merge(pm.double().numpy(), pl.double().numpy(), po.double().numpy())
    torch.cuda.synchronize()
    check_attn(f64(o), On, "merged O")
    check_attn(f64(lse), rlse, "merged lse")
    # fp32 partials merged in fp32: lse within 1e-4 (the exp2 of differences
    # of fp32 maxima and the fp32 sums stay far below it)
    check_lse_tight(f64(lse), rlse, 1e-4, "merged lse (tight)")
    assert f64(o)[0].max() == 0.0 and f64(o)[0].min() == 0.0 and np.isneginf(f64(lse)[0])
    assert np.isneginf(f64(m)[0]) and f64(l)[0] == 0.0
    fin = np.isfinite(rm)
    np.testing.assert_allclose(f64(m)[fin], rm[fin], rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(f64(l)[fin], rl[fin], rtol=1e-5)


@pytest.mark.parametrize("S", [3, 16])
def test_merge_unnormalised_nests(S):
    # merging in two stages (halves, then the two results) equals one merge
    pm, pl, po = random_partials(20, 2 * S, 128, seed=77 + S)
    o1, m1, l1, _ = oss.merge_partials(pm[:, :S].contiguous().cuda(), pl[:, :S].contiguous().cuda(),
                                       po[:, :S].contiguous().cuda(), finalize=False)
    o2, m2, l2, _ = oss.merge_partials(pm[:, S:].contiguous().cuda(), pl[:, S:].contiguous().cuda(),
                                       po[:, S:].contiguous().cuda(), finalize=False)
    o, m, l, lse = oss.merge_partials(torch.stack([m1, m2], 1), torch.stack([l1, l2], 1),
                                      torch.stack([o1, o2], 1), finalize=True)
    On, rm, rl, rlse = oracle.merge(pm.double().numpy(), pl.double().numpy(), po.double().numpy())
    torch.cuda.synchronize()
    check_attn(f64(o), On, "nested O")
    check_attn(f64(lse), rlse, "nested lse")
    Ou = oracle.merge(pm[:, :S].double().numpy(), pl[:, :S].double().numpy(),
                      po[:, :S].double().numpy(), finalize=False)[2]
    np.testing.assert_allclose(f64(o1), Ou, rtol=1e-5, atol=1e-4)
