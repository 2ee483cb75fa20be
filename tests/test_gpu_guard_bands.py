"""Canary guard bands around every output of the attention forward, its
partial-state form, split-KV decode and the merge (GPU).

Each output is a view into a larger buffer whose elements before and after
it -- and, for the partial-state arrays, the slots of the other shards -- are
filled with a canary bit pattern. After the call the canaries must be intact
bit for bit and the output itself must match the oracle. This stands in for
a memory checker: a stray store outside an output's extent changes a canary.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import pass_attention_gb300 as oss
from pass_attention_gb300 import workloads
from parity import check_attn

pytestmark = pytest.mark.gpu

PAD = 4096  # elements of canary on each side (a multiple of 16 bytes for every dtype)
CANARY = {torch.float32: 0x7FA5A5A5, torch.bfloat16: 0x7FA5}   # NaN payloads no kernel writes


def f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def banded(shape, dtype):
    """(buffer, view): the view has `shape` and sits PAD elements into a
    canary-filled buffer with PAD elements after it."""
    n = int(np.prod(shape))
    int_t = torch.int32 if dtype == torch.float32 else torch.int16
    raw = torch.full((n + 2 * PAD,), CANARY[dtype], dtype=torch.int64, device="cuda")
    if dtype == torch.bfloat16:
        raw = raw.to(torch.int16)
    else:
        raw = raw.to(torch.int32)
    buf = raw.view(dtype)
    assert buf.dtype == dtype and raw.dtype == int_t
    return buf, buf[PAD:PAD + n].view(shape)


def bands_intact(buf, what):
    raw = buf.view(torch.int32 if buf.dtype == torch.float32 else torch.int16)
    canary = torch.tensor(CANARY[buf.dtype], dtype=torch.int64).to(raw.dtype).item()
    head, tail = raw[:PAD], raw[-PAD:]
    assert bool((head == canary).all()), f"{what}: store before the output"
    assert bool((tail == canary).all()), f"{what}: store after the output"


@pytest.mark.parametrize("B,H,Sq,Sk,causal", [(2, 3, 300, 200, False), (1, 2, 300, 300, True),
                                               (1, 1, 1, 1, False), (2, 2, 129, 129, True)])
def test_attention_outputs_banded(B, H, Sq, Sk, causal):
    q, k, v = workloads.qkv(B, H, Sq, Sk, 128, seed=Sq + 7 * Sk, device="cuda")
    ob, o = banded((B, H, Sq, 128), torch.bfloat16)
    lb, lse = banded((B, H, Sq), torch.float32)
    scale = 1.0 / math.sqrt(128)
    oss.attention_fwd(q, k, v, scale, causal, o=o, lse=lse)
    assert oss.check_device_error() == 0
    bands_intact(ob, "o")
    bands_intact(lb, "lse")
    O, L = oracle.attention(f64(q), f64(k), f64(v), scale, causal)
    check_attn(f64(o), O, "o")
    check_attn(f64(lse), L, "lse")


@pytest.mark.parametrize("stride,index", [(4, 1), (3, 0), (5, 3)])
def test_attention_partial_slots_banded(stride, index):
    # index < stride - 1: the slots of the other shards and the bands around
    # the arrays keep their canaries
    B, H, Sq, Sk = 1, 3, 200, 300
    q, k, v = workloads.qkv(B, H, Sq, Sk, 128, seed=stride * 10 + index, device="cuda")
    mb, pm = banded((B, H, Sq, stride), torch.float32)
    lb, pl = banded((B, H, Sq, stride), torch.float32)
    obuf, po = banded((B, H, Sq, stride, 128), torch.float32)
    scale = 1.0 / math.sqrt(128)
    oss.attention_fwd_partial(q, k, v, pm, pl, po, index, scale)
    assert oss.check_device_error() == 0
    for buf, what in ((mb, "part_m"), (lb, "part_l"), (obuf, "part_o")):
        bands_intact(buf, what)
    canary32 = np.array([CANARY[torch.float32]], dtype=np.uint32)
    others = [s for s in range(stride) if s != index]
    for t, what in ((pm, "part_m"), (pl, "part_l"), (po, "part_o")):
        bits = t.cpu().numpy().view(np.uint32)
        assert np.all(bits[:, :, :, others] == canary32[0]), f"{what}: another shard's slot written"
    O, L = oracle.attention(f64(q), f64(k), f64(v), scale, False)
    pmh, plh, poh = f64(pm)[..., index], f64(pl)[..., index], f64(po)[..., index, :]
    check_attn(pmh + np.log(plh), L, "partial lse")
    check_attn(poh / plh[..., None], O, "partial O/l")


@pytest.mark.parametrize("S", [1, 7, 16])
def test_decode_partials_banded(S):
    B, H, Lmax = 3, 2, 400
    q, k, v, kv = workloads.decode_inputs(B, H, Lmax, 128, seed=S, device="cuda",
                                          kv_len=torch.tensor([400, 5, 123]))
    mb, pm = banded((B, H, S), torch.float32)
    lb, pl = banded((B, H, S), torch.float32)
    obuf, po = banded((B, H, S, 128), torch.float32)
    scale = 1.0 / math.sqrt(128)
    oss.attention_decode_splitkv(q, k, v, kv, S, scale, pm, pl, po)
    torch.cuda.synchronize()
    for buf, what in ((mb, "part_m"), (lb, "part_l"), (obuf, "part_o")):
        bands_intact(buf, what)
    rm, rl, ro = oracle.decode_partials(f64(q), f64(k), f64(v), kv.cpu().numpy(), S, scale)
    full = np.isfinite(rm)
    check_attn(f64(pm)[full] + np.log(f64(pl)[full]), rm[full] + np.log(rl[full]), "decode lse")


@pytest.mark.parametrize("finalize", [True, False])
@pytest.mark.parametrize("D", [4, 128, 256])
def test_merge_outputs_banded(finalize, D):
    G, S = 37, 5
    g = torch.Generator().manual_seed(D + int(finalize))
    pm = (torch.randn(G, S, generator=g, dtype=torch.float64) * 5)
    pl = torch.rand(G, S, generator=g, dtype=torch.float64) * 9 + 1
    po = torch.randn(G, S, D, generator=g, dtype=torch.float64)
    pm[3] = -math.inf
    pl[3] = 0.0
    po[3] = 0.0
    o_dtype = torch.bfloat16 if finalize else torch.float32
    obuf, o = banded((G, D), o_dtype)
    mb, m = banded((G,), torch.float32)
    lb, l = banded((G,), torch.float32)
    eb, lse = banded((G,), torch.float32)
    oss.merge_partials(pm.float().cuda(), pl.float().cuda(), po.float().cuda(), finalize,
                       o_out=o, m_out=m, l_out=l, lse_out=lse)
    torch.cuda.synchronize()
    for buf, what in ((obuf, "o_out"), (mb, "m_out"), (lb, "l_out"), (eb, "lse_out")):
        bands_intact(buf, what)
    On, rm, rl, rlse = oracle.merge(pm.float().double().numpy(), pl.float().double().numpy(),
                                    po.float().double().numpy())
    if finalize:
        check_attn(f64(o), On, "merged O")
    check_attn(f64(lse), rlse, "merged lse")


def test_binding_refuses_wrong_outputs():
    # outputs of the wrong length, shape, type or place are refused before
    # the library is called
    x = torch.zeros(4, 64, device="cuda")
    with pytest.raises(ValueError):
        oss.softmax_rows(x, m=torch.empty(3, device="cuda"))
    with pytest.raises(ValueError):
        oss.softmax_rows(x, l=torch.empty(4))
    with pytest.raises(TypeError):
        oss.softmax_rows_16bit(x.bfloat16(), m=torch.empty(4, device="cuda", dtype=torch.float16))
    with pytest.raises(ValueError):
        oss.softmax_rows_multipass(x, 2, l=torch.empty(8, device="cuda")[::2])
    q = torch.zeros(1, 2, 64, 128, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        oss.attention_fwd(q, q, q, o=torch.empty(1, 2, 63, 128, device="cuda", dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        oss.attention_fwd(q, q, q, lse=torch.empty(1, 2, 63, device="cuda"))
    with pytest.raises(ValueError):
        oss.attention_fwd(q, q, q, lse=torch.empty(1, 2, 64))
    pm = torch.empty(1, 2, 64, 2, device="cuda")
    po = torch.empty(1, 2, 64, 2, 128, device="cuda")
    with pytest.raises(ValueError):
        oss.attention_fwd_partial(q, q, q, pm, pm[..., :1].contiguous(), po, 0)
    with pytest.raises(ValueError):
        oss.attention_fwd_partial(q, q, q, pm, pm.clone(), po, 2)
    qd = torch.zeros(1, 2, 128, device="cuda", dtype=torch.bfloat16)
    kd = torch.zeros(1, 2, 32, 128, device="cuda", dtype=torch.bfloat16)
    kv = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        oss.attention_decode_splitkv(qd, kd, kd, kv, 4, part_m=torch.empty(1, 2, 3, device="cuda"))
    with pytest.raises(ValueError):
        oss.attention_decode_splitkv(qd, kd, kd, kv, 4, part_o=torch.empty(1, 2, 4, 64, device="cuda"))
    with pytest.raises(ValueError):
        oss.attention_decode_splitkv(qd, kd, kd, torch.ones(1, dtype=torch.int32), 4)
    mp = torch.zeros(5, 3, device="cuda")
    op = torch.zeros(5, 3, 8, device="cuda")
    with pytest.raises(TypeError):
        oss.merge_partials(mp, mp, op, True, o_out=torch.empty(5, 8, device="cuda"))
    with pytest.raises(ValueError):
        oss.merge_partials(mp, mp, op, False, o_out=torch.empty(5, 7, device="cuda"))
    with pytest.raises(ValueError):
        oss.merge_partials(mp, mp, op, lse_out=torch.empty(4, device="cuda"))
    with pytest.raises(ValueError):
        oss.merge_partials(mp, mp, op, m_out=torch.empty(5))
